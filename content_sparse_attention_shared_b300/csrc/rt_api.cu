// C-ABI layer: argument validation, workspace carving and the launch order of
// the routing-attention pass.  No allocation, no synchronisation and no host
// copies happen in the compute entry points.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "rt_internal.cuh"

namespace rt {

// ---------------------------------------------------------------------------
// launch counting and the per-launch timing hook
// ---------------------------------------------------------------------------
static std::atomic<long long> g_launches{0};
static std::mutex g_prof_mu;
static std::vector<cudaEvent_t> g_prof_events;
static std::vector<int> g_prof_kinds;
static int g_prof_pairs = 0;
static int g_prof_next = 0;
static thread_local int t_prof_slot = -1;

// A timing event around a launch.  Under stream capture it becomes an event
// record node of the graph (recorded at every replay) rather than a
// capture-time dependency, so a captured step can be timed kernel by kernel.
static cudaError_t record_timing_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
    cudaGetLastError();
    st = cudaStreamCaptureStatusNone;
  }
  return st == cudaStreamCaptureStatusActive
             ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
             : cudaEventRecord(ev, s);
}

void launch_begin(int kind, cudaStream_t s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  t_prof_slot = -1;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (g_prof_next < g_prof_pairs) {
    t_prof_slot = g_prof_next++;
    g_prof_kinds[t_prof_slot] = kind;
    if (record_timing_event(g_prof_events[2 * t_prof_slot], s) != cudaSuccess) {
      cudaGetLastError();  // a bad timing event must not fail the launch
      g_prof_kinds[t_prof_slot] = -1;
    }
  }
}

void launch_end(int kind, cudaStream_t s) {
  (void)kind;
  if (t_prof_slot < 0) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (t_prof_slot < g_prof_pairs &&
      record_timing_event(g_prof_events[2 * t_prof_slot + 1], s) != cudaSuccess)
    cudaGetLastError();
  t_prof_slot = -1;
}

// ---------------------------------------------------------------------------
// the device-side timeout test aid (rt_debug_inject_wait_timeout)
// ---------------------------------------------------------------------------
static std::atomic<unsigned> g_fault_kinds{0};
static std::atomic<unsigned long long> g_fault_ns{0};

uint64_t injected_limit_ns(int kind) {
  const unsigned kinds = g_fault_kinds.load(std::memory_order_relaxed);
  unsigned bit = 0;
  if (kind == K_SCORE_TC) bit = RT_DEBUG_SCORE;
  else if (kind == K_ATTN_TC) bit = RT_DEBUG_ATTENTION;
  else if (kind == K_LOCAL_ATTN) bit = RT_DEBUG_LOCAL_ATTENTION;
  return (kinds & bit) ? (uint64_t)g_fault_ns.load(std::memory_order_relaxed) : 0;
}

// ---------------------------------------------------------------------------
// dynamic shared-memory limits, set once per (kernel, device)
// ---------------------------------------------------------------------------
static std::mutex g_attr_mu;
static std::map<std::pair<const void*, int>, int> g_attr_set;

cudaError_t set_smem_limit(const void* func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  auto key = std::make_pair(func, dev);
  auto it = g_attr_set.find(key);
  if (it != g_attr_set.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) g_attr_set[key] = bytes;
  return e;
}

// ---------------------------------------------------------------------------
// the side stream of the training step (one per device, created on first use)
// ---------------------------------------------------------------------------
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
static std::mutex g_side_mu;  // held from the fork to the join of a step
static std::map<int, SideStream> g_side;

static cudaError_t side_stream(SideStream* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  auto it = g_side.find(dev);
  if (it == g_side.end()) {
    SideStream ss;
    e = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
    it = g_side.emplace(dev, ss).first;
  }
  *out = it->second;
  return cudaSuccess;
}

// ---------------------------------------------------------------------------
// tensor maps (cuTensorMapEncodeTiled through the runtime's driver entry
// point), with a small cache
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
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

bool tensor_maps_available() { return encode_fn() != nullptr; }

bool bf16_tensor_map_2d(const void* base, unsigned long long rows, unsigned cols,
                        unsigned box_cols, unsigned box_rows, CUtensorMap* out) {
  struct Entry {
    const void* ptr;
    unsigned long long rows;
    unsigned cols, box_cols, box_rows;
    CUtensorMap map;
  };
  constexpr int N = 16;
  static std::mutex mu;
  static Entry cache[N];
  static int used = 0, next = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].ptr == base && cache[i].rows == rows && cache[i].cols == cols &&
          cache[i].box_cols == box_cols && cache[i].box_rows == box_rows) {
        *out = cache[i].map;
        return true;
      }
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc || box_cols * 2 != 128) return false;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lk(mu);
  cache[next] = Entry{base, rows, cols, box_cols, box_rows, map};
  next = (next + 1) % N;
  if (used < N) ++used;
  *out = map;
  return true;
}

bool f32_tensor_map_3d(const void* base, unsigned cols, unsigned long long rows,
                       unsigned batches, unsigned box_rows, CUtensorMap* out) {
  struct Entry {
    const void* ptr;
    unsigned long long rows;
    unsigned cols, batches, box_rows;
    CUtensorMap map;
  };
  constexpr int N = 16;
  static std::mutex mu;
  static Entry cache[N];
  static int used = 0, next = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].ptr == base && cache[i].rows == rows && cache[i].cols == cols &&
          cache[i].batches == batches && cache[i].box_rows == box_rows) {
        *out = cache[i].map;
        return true;
      }
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc || cols % 32 != 0 || box_rows < 1 || box_rows > 256) return false;
  CUtensorMap map;
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)batches};
  const cuuint64_t strides[2] = {(cuuint64_t)cols * 4, (cuuint64_t)cols * 4 * rows};
  const cuuint32_t box[3] = {32u, (cuuint32_t)box_rows, 1u};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lk(mu);
  cache[next] = Entry{base, rows, cols, batches, box_rows, map};
  next = (next + 1) % N;
  if (used < N) ++used;
  *out = map;
  return true;
}

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------
static inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct FwdLayout {
  size_t err, S, gbins, mcount, slots, idx, assign, yslot, prep, idx_k, mvis, ema, total;
};

static FwdLayout fwd_layout(int B, int H, int n, int d, int k, int w, rt_dtype dt) {
  const size_t BH = (size_t)B * H;
  FwdLayout L;
  size_t off = 0;
  L.err = off; off += 256;
  L.S = off; off += align256(BH * k * n * sizeof(float));
  L.gbins = off;
  if (select_wants_group_bins(n)) off += align256(BH * k * (size_t)gbin_stride(n) * sizeof(uint16_t));
  L.mcount = off; off += align256(BH * n * sizeof(int32_t));
  L.slots = off; off += align256(BH * n * SLOTS_PER_ROW * sizeof(int32_t));
  L.idx = off; off += align256(BH * k * w * sizeof(int32_t));
  L.assign = off; off += align256(BH * n * sizeof(int32_t));
  L.yslot = off; off += align256(BH * k * w * d * sizeof(float));
  L.prep = off; off += align256(score_prep_bytes(H, d, k));
  L.idx_k = off; off += align256(BH * k * w * sizeof(int32_t));   // separate QK only
  L.mvis = off; off += align256(BH * n * sizeof(int32_t));        // separate QK only
  L.ema = off; off += align256(ema_workspace_bytes(B, H, n, d, k, dt));  // the training step
  L.total = off;
  return L;
}

struct BwdLayout {
  size_t err, mcount, slots, dq_slot, dv_slot, total;
};

static BwdLayout bwd_layout(int B, int H, int n, int d, int k, int w) {
  const size_t BH = (size_t)B * H;
  BwdLayout L;
  size_t off = 0;
  L.err = off; off += 256;
  L.mcount = off; off += align256(BH * n * sizeof(int32_t));
  L.slots = off; off += align256(BH * n * SLOTS_PER_ROW * sizeof(int32_t));
  L.dq_slot = off; off += align256(BH * k * w * d * sizeof(float));
  L.dv_slot = off; off += align256(BH * k * w * d * sizeof(float));
  L.total = off;
  return L;
}

static size_t ema_total(int B, int H, int n, int d, int k, rt_dtype dt) {
  return 256 + ema_workspace_bytes(B, H, n, d, k, dt);
}

}  // namespace rt

using namespace rt;

// ---------------------------------------------------------------------------
// error reporting
// ---------------------------------------------------------------------------
static thread_local char t_err[512];

static rt_status fail(rt_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
  return s;
}

static rt_status ok() {
  t_err[0] = '\0';
  return RT_OK;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static rt_status check_shape(rt_dtype dt, int B, int H, int n, int d, int k, int w) {
  if (dt != RT_F32 && dt != RT_BF16) return fail(RT_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (B < 1 || H < 1 || n < 1 || k < 1 || w < 1)
    return fail(RT_ERR_INVALID_ARG, "sizes must be positive (B=%d H=%d n=%d k=%d w=%d)", B, H, n, k, w);
  if (w > n) return fail(RT_ERR_INVALID_ARG, "w=%d exceeds n=%d", w, n);
  if (d != 64 && d != 128) return fail(RT_ERR_UNSUPPORTED, "head dimension d=%d (supported: 64, 128)", d);
  const double bhkn = (double)B * H * k * n;
  const double bhkwd = (double)B * H * k * w * d;
  if (bhkn > 4.0e9 || bhkwd > 1.6e10 || (double)B * H * n * d > 1.6e10)
    return fail(RT_ERR_UNSUPPORTED, "problem too large for one call");
  if ((double)B * n > 12.0e6) return fail(RT_ERR_UNSUPPORTED, "B*n above 12M rows per head");
  return RT_OK;
}

static rt_status from_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return RT_OK;
  return fail(RT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

extern "C" {

const char* rt_status_string(rt_status s) {
  switch (s) {
    case RT_OK: return "RT_OK";
    case RT_ERR_INVALID_ARG: return "RT_ERR_INVALID_ARG";
    case RT_ERR_UNSUPPORTED: return "RT_ERR_UNSUPPORTED";
    case RT_ERR_WORKSPACE: return "RT_ERR_WORKSPACE";
    case RT_ERR_CUDA: return "RT_ERR_CUDA";
    case RT_ERR_TIMEOUT: return "RT_ERR_TIMEOUT";
  }
  return "RT_ERR_UNKNOWN";
}

const char* rt_last_error_detail(void) { return t_err; }

int64_t rt_launch_count(void) { return (int64_t)g_launches.load(); }

rt_status rt_debug_inject_wait_timeout(unsigned kernels, unsigned long long limit_ns) {
  if (kernels & ~(unsigned)(RT_DEBUG_SCORE | RT_DEBUG_ATTENTION | RT_DEBUG_LOCAL_ATTENTION))
    return fail(RT_ERR_INVALID_ARG, "unknown kernel bits 0x%x", kernels);
  if (kernels != 0 && (limit_ns == 0 || limit_ns > 1000000000ull))
    return fail(RT_ERR_INVALID_ARG, "limit_ns must be in (0, 1e9]");
  g_fault_ns.store(kernels ? limit_ns : 0ull);
  g_fault_kinds.store(kernels);
  return ok();
}

rt_status rt_profile_set(void* const* events, int n_pairs) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (n_pairs < 0 || (n_pairs > 0 && events == nullptr))
    return fail(RT_ERR_INVALID_ARG, "bad profile event array");
  g_prof_events.assign(2 * (size_t)n_pairs, nullptr);
  for (int i = 0; i < 2 * n_pairs; ++i) g_prof_events[i] = static_cast<cudaEvent_t>(events[i]);
  g_prof_kinds.assign(n_pairs, -1);
  g_prof_pairs = n_pairs;
  g_prof_next = 0;
  return ok();
}

int rt_profile_kernel_id(int i) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (i < 0 || i >= g_prof_next) return -1;
  return g_prof_kinds[i];
}

const char* rt_kernel_name(int id) {
  static const char* names[K_NUM_KINDS] = {
      "score_simt", "score_tc", "select_topw", "attention_simt", "attention_tc",
      "scatter_average", "ema_topw", "ema_update", "centroid_prep", "local_attention",
      "ema_bucket", "backward", "membership"};
  if (id < 0 || id >= K_NUM_KINDS) return "unknown";
  return names[id];
}

size_t rt_workspace_bytes(int B, int H, int n, int d, int k, int w, rt_dtype dt) {
  if (check_shape(dt, B, H, n, d, k, w) != RT_OK) return 0;
  const size_t a = fwd_layout(B, H, n, d, k, w, dt).total;
  const size_t b = ema_total(B, H, n, d, k, dt);
  const size_t c = bwd_layout(B, H, n, d, k, w).total;
  return std::max(a, std::max(b, c));
}

rt_status rt_route_assign(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                          const float* centroids, int k, int w, int32_t* idx, int32_t* assign,
                          float* scores, void* workspace, size_t workspace_bytes, void* stream) {
  rt_status st = check_shape(dt, B, H, n, d, k, w);
  if (st != RT_OK) return st;
  if (!qk || !centroids || !idx) return fail(RT_ERR_INVALID_ARG, "null qk/centroids/idx");
  if (!aligned16(qk) || !aligned16(centroids) || !aligned16(idx) ||
      (assign && !aligned16(assign)) || (scores && !aligned16(scores)))
    return fail(RT_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  const FwdLayout L = fwd_layout(B, H, n, d, k, w, dt);
  if (!workspace || workspace_bytes < L.total)
    return fail(RT_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes, L.total);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(RT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  float* S = scores ? scores : reinterpret_cast<float*>(ws + L.S);
  unsigned int* err = reinterpret_cast<unsigned int*>(ws + L.err);
  void* prep = score_prep_bytes(H, d, k) ? static_cast<void*>(ws + L.prep) : nullptr;
  uint16_t* gbins =
      select_wants_group_bins(n) ? reinterpret_cast<uint16_t*>(ws + L.gbins) : nullptr;
  st = from_cuda(
      launch_score(qk, dt, B, H, n, d, centroids, k, S, assign, nullptr, gbins, prep, err, s),
      "score kernel");
  if (st != RT_OK) return st;
  st = from_cuda(launch_select(S, gbins, BH, n, k, w, idx, nullptr, nullptr, s), "select kernel");
  if (st != RT_OK) return st;
  return ok();
}

// The forward pass for both forms.  Shared QK (kp == q): score, select,
// attention on the packed / key-block kernels, scatter.  Separate keys: the
// queries and the keys are each scored and selected against the same
// centroids, the key-block kernel attends between a cluster's queries and its
// keys with the mask on original positions, and the scatter divides by each
// position's count of memberships with a visible key.
// The centroid step a training step adds to the forward pass (mu == nullptr:
// none).  It needs only the argmax assignment, so it is forked onto the side
// stream right after the score kernel and runs beside the select, attention
// and scatter kernels (all latency-bound); the pass joins it back at its end.
// (Forking after the attention kernel instead, beside the scatter only,
// measured 3 us slower at n = 8192.)
struct StepEma {
  float* mu = nullptr;
  float decay = 0.0f;
};

static rt_status forward(const void* q, const void* kp, const void* v, rt_dtype dt, int B, int H,
                         int n, int d, const float* centroids, int kc, int w, int causal,
                         float scale, void* out, int32_t* idx_out, int32_t* idx_k_out,
                         int32_t* assign_out, void* workspace, size_t workspace_bytes,
                         void* stream, const StepEma& ema = StepEma()) {
  rt_status st = check_shape(dt, B, H, n, d, kc, w);
  if (st != RT_OK) return st;
  if (!q || !kp || !v || !centroids || !out) return fail(RT_ERR_INVALID_ARG, "null tensor pointer");
  if (causal != 0 && causal != 1) return fail(RT_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!std::isfinite(scale)) return fail(RT_ERR_INVALID_ARG, "scale is not finite");
  if (!aligned16(q) || !aligned16(kp) || !aligned16(v) || !aligned16(centroids) ||
      !aligned16(out) || (idx_out && !aligned16(idx_out)) ||
      (idx_k_out && !aligned16(idx_k_out)) || (assign_out && !aligned16(assign_out)))
    return fail(RT_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  const FwdLayout L = fwd_layout(B, H, n, d, kc, w, dt);
  if (!workspace || workspace_bytes < L.total)
    return fail(RT_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes, L.total);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(RT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (scale <= 0.0f) scale = 1.0f / sqrtf((float)d);
  const bool separate = kp != q;

  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  float* S = reinterpret_cast<float*>(ws + L.S);
  int32_t* mcount = reinterpret_cast<int32_t*>(ws + L.mcount);
  int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(ws + L.idx);
  float* yslot = reinterpret_cast<float*>(ws + L.yslot);
  int32_t* slots = reinterpret_cast<int32_t*>(ws + L.slots);
  unsigned int* err = reinterpret_cast<unsigned int*>(ws + L.err);
  void* prep = score_prep_bytes(H, d, kc) ? static_cast<void*>(ws + L.prep) : nullptr;

  int32_t* assign = assign_out;
  if (ema.mu != nullptr && assign == nullptr) assign = reinterpret_cast<int32_t*>(ws + L.assign);
  std::unique_lock<std::mutex> side_lock(g_side_mu, std::defer_lock);
  SideStream side;
  if (ema.mu != nullptr) {
    side_lock.lock();
    st = from_cuda(side_stream(&side), "creating the side stream");
    if (st != RT_OK) return st;
  }
  auto fork_ema = [&]() -> rt_status {
    cudaError_t e = cudaEventRecord(side.fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side.s, side.fork, 0);
    if (e == cudaSuccess)
      e = launch_ema(q, dt, B, H, n, d, assign, ema.mu, kc, ema.decay, ws + L.ema, side.s);
    if (e == cudaSuccess) e = cudaEventRecord(side.join, side.s);
    return from_cuda(e, "centroid update (side stream)");
  };

  uint16_t* gbins =
      select_wants_group_bins(n) ? reinterpret_cast<uint16_t*>(ws + L.gbins) : nullptr;
  st = from_cuda(
      launch_score(q, dt, B, H, n, d, centroids, kc, S, assign, mcount, gbins, prep, err, s),
      "score kernel");
  if (st != RT_OK) return st;
  if (ema.mu != nullptr) {
    st = fork_ema();
    if (st != RT_OK) return st;
  }
  st = from_cuda(launch_select(S, gbins, BH, n, kc, w, idx, mcount, slots, s), "select kernel");
  if (st != RT_OK) return st;
  int32_t* idx_k = nullptr;
  int32_t* mvis = nullptr;
  if (separate) {
    idx_k = idx_k_out ? idx_k_out : reinterpret_cast<int32_t*>(ws + L.idx_k);
    mvis = reinterpret_cast<int32_t*>(ws + L.mvis);
    // the keys' routing; the score kernel zeroes mvis for the attention
    st = from_cuda(
        launch_score(kp, dt, B, H, n, d, centroids, kc, S, nullptr, mvis, gbins, prep, err, s),
        "score kernel (keys)");
    if (st != RT_OK) return st;
    st = from_cuda(launch_select(S, gbins, BH, n, kc, w, idx_k, nullptr, nullptr, s),
                   "select kernel (keys)");
    if (st != RT_OK) return st;
    if (attention_tc_supported(dt, d, w)) {
      st = from_cuda(launch_attention_separate_tc(q, kp, v, BH, n, d, kc, w, causal, scale, idx,
                                                  idx_k, mcount, mvis, out, yslot, err, s),
                     "attention kernel");
    } else {
      st = from_cuda(launch_attention_simt(q, kp, v, dt, BH, n, d, kc, w, causal, scale, idx,
                                           idx_k, mcount, mvis, out, yslot, s),
                     "attention kernel");
    }
  } else if (attention_tc_supported(dt, d, w)) {
    st = from_cuda(launch_attention_tc(q, v, BH, n, d, kc, w, causal, scale, idx, mcount, out,
                                       yslot, err, s),
                   "attention kernel");
  } else {
    st = from_cuda(launch_attention_simt(q, kp, v, dt, BH, n, d, kc, w, causal, scale, idx,
                                         nullptr, mcount, nullptr, out, yslot, s),
                   "attention kernel");
  }
  if (st != RT_OK) return st;
  st = from_cuda(launch_scatter(dt, BH, n, d, kc, w, idx, mcount, mvis, slots, yslot, out, s),
                 "scatter kernel");
  if (st != RT_OK) return st;
  if (ema.mu != nullptr) {
    st = from_cuda(cudaStreamWaitEvent(s, side.join, 0), "joining the side stream");
    if (st != RT_OK) return st;
  }
  return ok();
}

rt_status rt_routing_attention(const void* q, const void* kp, const void* v, rt_dtype dt, int B,
                               int H, int n, int d, const float* centroids, int kc, int w,
                               int causal, float scale, void* out, int32_t* idx_out,
                               int32_t* assign_out, void* workspace, size_t workspace_bytes,
                               void* stream) {
  return forward(q, kp, v, dt, B, H, n, d, centroids, kc, w, causal, scale, out, idx_out,
                 nullptr, assign_out, workspace, workspace_bytes, stream);
}

rt_status rt_routing_attention_step(const void* q, const void* v, rt_dtype dt, int B, int H,
                                    int n, int d, float* centroids, int kc, int w, int causal,
                                    float scale, float decay, void* out, int32_t* idx_out,
                                    int32_t* assign_out, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  if (!(decay >= 0.0f && decay <= 1.0f)) return fail(RT_ERR_INVALID_ARG, "decay must be in [0, 1]");
  if (kc > 4096) return fail(RT_ERR_UNSUPPORTED, "k above 4096 for the centroid update");
  if (!centroids) return fail(RT_ERR_INVALID_ARG, "null centroids");
  StepEma ema;
  ema.mu = centroids;
  ema.decay = decay;
  return forward(q, q, v, dt, B, H, n, d, centroids, kc, w, causal, scale, out, idx_out, nullptr,
                 assign_out, workspace, workspace_bytes, stream, ema);
}

rt_status rt_routing_attention_separate(const void* q, const void* kp, const void* v, rt_dtype dt,
                                        int B, int H, int n, int d, const float* centroids,
                                        int kc, int w, int causal, float scale, void* out,
                                        int32_t* idx_q_out, int32_t* idx_k_out,
                                        int32_t* assign_out, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  if (q != nullptr && q == kp)
    return fail(RT_ERR_INVALID_ARG, "separate keys: k must be a different tensor from q "
                                    "(rt_routing_attention takes shared QK)");
  return forward(q, kp, v, dt, B, H, n, d, centroids, kc, w, causal, scale, out, idx_q_out,
                 idx_k_out, assign_out, workspace, workspace_bytes, stream);
}

rt_status rt_routing_attention_backward(const void* q, const void* v, rt_dtype dt, int B, int H,
                                        int n, int d, const int32_t* idx, int kc, int w,
                                        int causal, float scale, const float* dout, float* dq,
                                        float* dv, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  rt_status st = check_shape(dt, B, H, n, d, kc, w);
  if (st != RT_OK) return st;
  if (!q || !v || !idx || !dout || !dq || !dv) return fail(RT_ERR_INVALID_ARG, "null tensor pointer");
  if (causal != 0 && causal != 1) return fail(RT_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!std::isfinite(scale)) return fail(RT_ERR_INVALID_ARG, "scale is not finite");
  if (!aligned16(q) || !aligned16(v) || !aligned16(idx) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dv))
    return fail(RT_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  const BwdLayout L = bwd_layout(B, H, n, d, kc, w);
  if (!workspace || workspace_bytes < L.total)
    return fail(RT_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes, L.total);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(RT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (scale <= 0.0f) scale = 1.0f / sqrtf((float)d);
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  unsigned int* err = reinterpret_cast<unsigned int*>(ws + L.err);
  int32_t* mcount = reinterpret_cast<int32_t*>(ws + L.mcount);
  int32_t* slots = reinterpret_cast<int32_t*>(ws + L.slots);
  float* dq_slot = reinterpret_cast<float*>(ws + L.dq_slot);
  float* dv_slot = reinterpret_cast<float*>(ws + L.dv_slot);
  st = from_cuda(launch_membership(idx, BH, n, kc, w, mcount, slots, s), "membership kernel");
  if (st != RT_OK) return st;
  st = from_cuda(launch_backward_clusters(q, v, dt, BH, n, d, kc, w, causal, scale, idx, mcount,
                                          dout, dq_slot, dv_slot, s),
                 "backward kernel");
  if (st != RT_OK) return st;
  st = from_cuda(launch_gather_sum(BH, n, d, kc, w, idx, mcount, slots, dq_slot, dq, s),
                 "gradient gather (dq)");
  if (st != RT_OK) return st;
  st = from_cuda(launch_gather_sum(BH, n, d, kc, w, idx, mcount, slots, dv_slot, dv, s),
                 "gradient gather (dv)");
  if (st != RT_OK) return st;
  return ok();
}

rt_status rt_centroid_ema(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                          const int32_t* assign, float* centroids, int k, float decay,
                          void* workspace, size_t workspace_bytes, void* stream) {
  rt_status st = check_shape(dt, B, H, n, d, k, 1);
  if (st != RT_OK) return st;
  if (!qk || !assign || !centroids) return fail(RT_ERR_INVALID_ARG, "null qk/assign/centroids");
  if (!(decay >= 0.0f && decay <= 1.0f)) return fail(RT_ERR_INVALID_ARG, "decay must be in [0, 1]");
  if (!aligned16(qk) || !aligned16(assign) || !aligned16(centroids))
    return fail(RT_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (k > 4096) return fail(RT_ERR_UNSUPPORTED, "k above 4096 for the centroid update");
  const size_t need = ema_total(B, H, n, d, k, dt);
  if (!workspace || workspace_bytes < need)
    return fail(RT_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes, need);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(RT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = from_cuda(launch_ema(qk, dt, B, H, n, d, assign, centroids, k, decay, ws + 256, s),
                 "centroid update kernels");
  if (st != RT_OK) return st;
  return ok();
}

rt_status rt_centroid_ema_sums(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                               const int32_t* assign, int k, float* sums, void* workspace,
                               size_t workspace_bytes, void* stream) {
  rt_status st = check_shape(dt, B, H, n, d, k, 1);
  if (st != RT_OK) return st;
  if (!qk || !assign || !sums) return fail(RT_ERR_INVALID_ARG, "null qk/assign/sums");
  if (!aligned16(qk) || !aligned16(assign) || !aligned16(sums))
    return fail(RT_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (k > 4096) return fail(RT_ERR_UNSUPPORTED, "k above 4096 for the centroid update");
  const size_t need = ema_total(B, H, n, d, k, dt);
  if (!workspace || workspace_bytes < need)
    return fail(RT_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes, need);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(RT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  char* ws = static_cast<char*>(workspace);
  st = from_cuda(launch_ema_sums(qk, dt, B, H, n, d, assign, k, sums, ws + 256,
                                 static_cast<cudaStream_t>(stream)),
                 "centroid sum kernels");
  if (st != RT_OK) return st;
  return ok();
}

rt_status rt_centroid_ema_apply(const float* sums, int H, int d, float* centroids, int k,
                                float decay, void* stream) {
  if (H < 1 || k < 1) return fail(RT_ERR_INVALID_ARG, "H and k must be positive");
  if (d != 64 && d != 128) return fail(RT_ERR_UNSUPPORTED, "head dimension d=%d (supported: 64, 128)", d);
  if (!sums || !centroids) return fail(RT_ERR_INVALID_ARG, "null sums/centroids");
  if (!(decay >= 0.0f && decay <= 1.0f)) return fail(RT_ERR_INVALID_ARG, "decay must be in [0, 1]");
  if (!aligned16(centroids) || (reinterpret_cast<uintptr_t>(sums) & 3u) != 0)
    return fail(RT_ERR_INVALID_ARG, "misaligned sums/centroids");
  if ((long long)H * k > 0x7fffffffLL) return fail(RT_ERR_UNSUPPORTED, "H*k too large");
  rt_status st = from_cuda(launch_ema_apply(sums, H, d, centroids, k, decay,
                                            static_cast<cudaStream_t>(stream)),
                           "centroid apply kernel");
  if (st != RT_OK) return st;
  return ok();
}

rt_status rt_centroid_ema_topw(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                               const int32_t* idx, int w, float* centroids, int k, float decay,
                               void* workspace, size_t workspace_bytes, void* stream) {
  rt_status st = check_shape(dt, B, H, n, d, k, w);
  if (st != RT_OK) return st;
  if (!qk || !idx || !centroids) return fail(RT_ERR_INVALID_ARG, "null qk/idx/centroids");
  if (!(decay >= 0.0f && decay <= 1.0f)) return fail(RT_ERR_INVALID_ARG, "decay must be in [0, 1]");
  if (!aligned16(qk) || !aligned16(idx) || !aligned16(centroids))
    return fail(RT_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (k > 4096) return fail(RT_ERR_UNSUPPORTED, "k above 4096 for the centroid update");
  const size_t need = ema_total(B, H, n, d, k, dt);
  if (!workspace || workspace_bytes < need)
    return fail(RT_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes, need);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(RT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  st = from_cuda(launch_ema_topw(qk, dt, B, H, n, d, idx, w, centroids, k, decay,
                                 static_cast<cudaStream_t>(stream)),
                 "top-w centroid update kernel");
  if (st != RT_OK) return st;
  return ok();
}

rt_status rt_local_attention(const void* q, const void* kp, const void* v, rt_dtype dt, int B,
                             int H, int n, int d, int window, float scale, void* out,
                             void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 1 || H < 1 || n < 1) return fail(RT_ERR_INVALID_ARG, "B, H and n must be positive");
  if (window < 1) return fail(RT_ERR_INVALID_ARG, "window must be at least 1");
  if (dt != RT_BF16 && dt != RT_F32) return fail(RT_ERR_INVALID_ARG, "unknown dtype");
  if (dt != RT_BF16) return fail(RT_ERR_UNSUPPORTED, "local attention takes bf16 rows");
  if (d != 64 && d != 128) return fail(RT_ERR_UNSUPPORTED, "d must be 64 or 128");
  if ((long long)B * H * n > 0x7fffffffLL) return fail(RT_ERR_UNSUPPORTED, "B*H*n too large");
  if (!q || !kp || !v || !out) return fail(RT_ERR_INVALID_ARG, "null tensor pointer");
  if (kp != q) return fail(RT_ERR_UNSUPPORTED, "separate keys: only shared QK (k == q)");
  if (!std::isfinite(scale)) return fail(RT_ERR_INVALID_ARG, "scale is not finite");
  if (!aligned16(q) || !aligned16(v) || !aligned16(out))
    return fail(RT_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (!workspace || workspace_bytes < 256)
    return fail(RT_ERR_WORKSPACE, "workspace %zu bytes, need 256", workspace_bytes);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(RT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (scale <= 0.0f) scale = 1.0f / sqrtf((float)d);
  unsigned int* err = static_cast<unsigned int*>(workspace);
  rt_status st = from_cuda(launch_local_attention(q, v, B * H, n, d, window, scale, out, err,
                                                  static_cast<cudaStream_t>(stream)),
                           "local attention kernel");
  if (st != RT_OK) return st;
  return ok();
}

rt_status rt_mixed_attention(const void* q, const void* v, rt_dtype dt, int B, int H, int n, int d,
                             int n_local, int window, const float* centroids, int kc, int w,
                             int causal, float scale, void* out, int32_t* idx_out,
                             int32_t* assign_out, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (B < 1 || H < 1 || n < 1) return fail(RT_ERR_INVALID_ARG, "B, H and n must be positive");
  if (n_local < 0 || n_local > H) return fail(RT_ERR_INVALID_ARG, "n_local=%d outside [0, H]", n_local);
  if (dt != RT_BF16 && dt != RT_F32) return fail(RT_ERR_INVALID_ARG, "unknown dtype");
  if (!q || !v || !out) return fail(RT_ERR_INVALID_ARG, "null tensor pointer");
  const int Hr = H - n_local;
  const size_t es = dt == RT_F32 ? 4 : 2;
  const size_t head = (size_t)n * d * es;  // bytes of one head of one sequence
  const size_t need = Hr > 0 ? rt_workspace_bytes(1, Hr, n, d, kc, w, dt) : 256;
  if (Hr > 0 && need == 0) return validate_shape(dt, 1, Hr, n, d, kc, w);
  if (Hr > 0 && !centroids) return fail(RT_ERR_INVALID_ARG, "null centroids");
  // both halves are checked here, before anything is launched
  if (n_local > 0) {
    if (dt != RT_BF16) return fail(RT_ERR_UNSUPPORTED, "local attention takes bf16 rows");
    if (window < 1) return fail(RT_ERR_INVALID_ARG, "window must be at least 1");
    if (d != 64 && d != 128) return fail(RT_ERR_UNSUPPORTED, "d must be 64 or 128");
  }
  if (Hr > 0 && (causal != 0 && causal != 1))
    return fail(RT_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!std::isfinite(scale)) return fail(RT_ERR_INVALID_ARG, "scale is not finite");
  if (!aligned16(q) || !aligned16(v) || !aligned16(out) || (centroids && !aligned16(centroids)) ||
      (idx_out && !aligned16(idx_out)) || (assign_out && !aligned16(assign_out)))
    return fail(RT_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (!workspace || workspace_bytes < need)
    return fail(RT_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes, need);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(RT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  for (int b = 0; b < B; ++b) {
    const char* qb = static_cast<const char*>(q) + (size_t)b * H * head;
    const char* vb = static_cast<const char*>(v) + (size_t)b * H * head;
    char* ob = static_cast<char*>(out) + (size_t)b * H * head;
    rt_status st;
    if (n_local > 0) {
      st = rt_local_attention(qb, qb, vb, dt, 1, n_local, n, d, window, scale, ob, workspace,
                              workspace_bytes, stream);
      if (st != RT_OK) return st;
    }
    if (Hr > 0) {
      const char* qr = qb + (size_t)n_local * head;
      st = rt_routing_attention(qr, qr, vb + (size_t)n_local * head, dt, 1, Hr, n, d, centroids,
                                kc, w, causal, scale, ob + (size_t)n_local * head,
                                idx_out ? idx_out + (size_t)b * Hr * kc * w : nullptr,
                                assign_out ? assign_out + (size_t)b * Hr * n : nullptr, workspace,
                                workspace_bytes, stream);
      if (st != RT_OK) return st;
    }
  }
  return ok();
}

rt_status rt_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < 256) return fail(RT_ERR_WORKSPACE, "no workspace");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(RT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  return from_cuda(cudaMemsetAsync(workspace, 0, 256, static_cast<cudaStream_t>(stream)),
                   "clearing the device status word") == RT_OK ? ok() : RT_ERR_CUDA;
}

rt_status rt_check_device_status(void* workspace, size_t workspace_bytes, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!workspace && workspace_bytes == 0) return noalloc_check_status(s);
  if (!workspace || workspace_bytes < 256) return fail(RT_ERR_WORKSPACE, "no workspace");
  unsigned int word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return from_cuda(e, "reading the device status word");
  if (word != DEV_OK) {
    const unsigned int zero = 0;
    e = cudaMemcpyAsync(workspace, &zero, sizeof(zero), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (word == DEV_TIMEOUT) return fail(RT_ERR_TIMEOUT, "a device-side wait ran out (code %u)", word);
    return fail(RT_ERR_CUDA, "device status word %u", word);
  }
  return ok();
}

}  // extern "C"

namespace rt {

rt_status record_error(rt_status s, const char* msg) {
  if (s == RT_OK) return ok();
  return fail(s, "%s", msg);
}

rt_status validate_shape(rt_dtype dt, int B, int H, int n, int d, int k, int w) {
  return check_shape(dt, B, H, n, d, k, w);
}

}  // namespace rt
