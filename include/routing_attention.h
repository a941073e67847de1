/*
 * routing_attention.h -- C ABI of the B300 (sm_103a) routing-attention library.
 *
 * Method: "Efficient Content-Based Sparse Attention with Routing Transformers"
 * (Roy, Saffar, Vaswani, Grangier; TACL 2021).  The pages describing it
 * (paperlayer.ai summary §4 "Efficient Content-Dependent Sparse Attention",
 * "Routing attention with clustering") fix the operation: queries and keys
 * are put on the unit sphere, routed to the nearest of k shared centroids
 * learned by online spherical k-means, and attention is computed only
 * between query/key pairs routed to the same cluster, with balanced clusters
 * of about n/k members.  The steps the pages leave open are read as follows
 * and implemented exactly so:
 *   - "unit-normalised" = subtract the row mean, divide by the Euclidean norm
 *     (a row with zero centred norm maps to the zero vector);
 *   - each centroid takes its own top-w tokens by score, ties to the lower
 *     position, and lists them in ascending position order;
 *   - attention inside a cluster uses the raw Q, K, V rows, scale 1/sqrt(d)
 *     unless given, causal on original positions (a token sees itself);
 *   - a token in several clusters receives the mean of its outputs, a token in
 *     none receives a zero row;
 *   - the centroid update blends the mean of the normalised rows assigned to
 *     each centroid (argmax assignment, over the whole batch) into the
 *     centroid with weight (1 - decay), then renormalises; a centroid with no
 *     assigned row is left unchanged (rt_centroid_ema_topw takes each
 *     centroid's own top-w lists instead of the argmax);
 *   - rt_local_attention is the sliding-window causal layer the pages pair
 *     with routing attention (a position sees the window ending at itself).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, contiguous,
 *     16-byte aligned, innermost dimension fastest.  Shapes are given in the
 *     argument comments ([B,H,n,d] means index ((b*H + h)*n + t)*d + j).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     Calls are asynchronous on that stream; the library never synchronises,
 *     never allocates device memory and never copies to the host inside the
 *     compute entry points.  All scratch lives in the caller's `workspace`
 *     of at least rt_workspace_bytes(...) bytes (256-byte aligned).
 *   - Errors found on the host (bad arguments, too-small workspace, a CUDA
 *     launch error) are returned immediately; nothing is launched then.
 *     A device-side error (a bounded wait that ran out) is recorded in the
 *     workspace and reported by rt_check_device_status().
 *   - Supported: d in {64, 128}; 1 <= w <= n; k >= 1; causal in {0, 1};
 *     dtype RT_F32 or RT_BF16 (Q, K, V and the output share it; centroids
 *     are always fp32).  Other values return RT_ERR_UNSUPPORTED or
 *     RT_ERR_INVALID_ARG.  There is no CPU fallback.
 */
#ifndef ROUTING_ATTENTION_H
#define ROUTING_ATTENTION_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rt_status {
  RT_OK = 0,
  RT_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer     */
  RT_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement    */
  RT_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required     */
  RT_ERR_CUDA = 4,         /* a CUDA call or kernel launch failed            */
  RT_ERR_TIMEOUT = 5       /* a device-side bounded wait ran out             */
} rt_status;

typedef enum rt_dtype { RT_F32 = 0, RT_BF16 = 1 } rt_dtype;

/* Bytes of device workspace the three compute calls need for this shape
 * (the maximum over them, so one buffer serves all).  Returns 0 for an
 * invalid shape. */
size_t rt_workspace_bytes(int B, int H, int n, int d, int k, int w, rt_dtype dt);

/* Routing only (steps: normalise, score, argmax, top-w per centroid, sort).
 * Source: §4 "Routing attention with clustering" (nearest-centroid routing
 * of unit-normalised shared queries/keys; balanced clusters via a top-k
 * assignment).
 *   qk        [B,H,n,d]  shared query/key rows (dtype dt)
 *   centroids [H,k,d]    fp32 centroids (read only)
 *   idx       [B,H,k,w]  out: the w positions chosen by each centroid,
 *                        strictly ascending
 *   assign    [B,H,n]    out, may be NULL: argmax centroid of every row
 *                        (ties to the lower centroid)
 *   scores    [B,H,k,n]  out, may be NULL: the fp32 scores <r_t, mu_c>
 */
rt_status rt_route_assign(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                          const float* centroids, int k, int w,
                          int32_t* idx, int32_t* assign, float* scores,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Full routing-attention forward pass: routing as above, dense softmax
 * attention inside every w-by-w cluster block (causal on original positions
 * when causal=1), and the averaging scatter back to positions.
 * Source: §3 "Self-Attentive Auto-regressive Sequence Modeling" (softmax
 * attention, causal masking) and §4 (same-cluster query/key pairs only).
 *   q, k, v   [B,H,n,d]  dtype dt; shared QK: k must equal q (the same
 *                        pointer), otherwise RT_ERR_UNSUPPORTED
 *   centroids [H,kc,d]   fp32 (read only; the update is rt_centroid_ema)
 *   scale     logit scale; <= 0 selects 1/sqrt(d)
 *   out       [B,H,n,d]  dtype dt; every row is written (zero rows for
 *                        positions no centroid chose)
 *   idx_out   [B,H,kc,w] out, may be NULL
 *   assign_out[B,H,n]    out, may be NULL (argmax centroid per row, the
 *                        input rt_centroid_ema expects)
 */
rt_status rt_routing_attention(const void* q, const void* k, const void* v, rt_dtype dt,
                               int B, int H, int n, int d,
                               const float* centroids, int kc, int w,
                               int causal, float scale,
                               void* out, int32_t* idx_out, int32_t* assign_out,
                               void* workspace, size_t workspace_bytes, void* stream);

/* One online spherical k-means step on the centroids, in place.
 * Source: §2 "Attention with Content-Based Sparsity" (centroids learned by
 * mini-batch spherical k-means), §4 (centroids shared across sequences,
 * learned online).  For every head h and centroid c:
 *   N = #{(b,t): assign[b,h,t] == c};  if N > 0:
 *   mu_c <- normalise(decay * mu_c + (1 - decay) * (1/N) * sum r_t)
 * with r_t the normalised row of qk; otherwise mu_c is left bit-exact.
 *   qk        [B,H,n,d]  dtype dt
 *   assign    [B,H,n]    int32 in [0, k)
 *   centroids [H,k,d]    fp32, updated in place
 *   decay     in [0, 1]
 * Each centroid's rows are listed in a fixed order and summed in that order,
 * with no floating-point atomics: results are deterministic.  Needs a
 * workspace of at least rt_workspace_bytes(B, H, n, d, k, 1, dt) bytes (only
 * its device status word is used). */
rt_status rt_centroid_ema(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                          const int32_t* assign, float* centroids, int k, float decay,
                          void* workspace, size_t workspace_bytes, void* stream);

/* The same step driven by the top-w membership instead of the argmax
 * assignment: centroid c of head h moves toward the normalised rows its own
 * lists chose.  The pages do not say which membership moves a centroid
 * (§4 "Routing attention with clustering": balanced clusters through a top-k
 * assignment, centroids learned online; §2: mini-batch spherical k-means);
 * rt_centroid_ema takes the argmax, this call the alternative.  For every
 * head h and centroid c:
 *   L = the entries t of idx[b,h,c,0..w) over every sequence b with 0 <= t < n
 *       (a position listed by several centroids counts for each of them);
 *   N = |L|;  if N > 0:
 *   mu_c <- normalise(decay * mu_c + (1 - decay) * (1/N) * sum_{t in L} r_t)
 * otherwise mu_c is left bit-exact.
 *   qk        [B,H,n,d]  dtype dt
 *   idx       [B,H,k,w]  int32, ascending per list (as rt_route_assign and
 *                        rt_routing_attention return it); other entries are
 *                        skipped
 *   centroids [H,k,d]    fp32, updated in place
 *   decay     in [0, 1]
 * Deterministic (rows summed in list order, no floating-point atomics).
 * Errors: RT_ERR_INVALID_ARG for null or misaligned pointers or decay out of
 * range, RT_ERR_UNSUPPORTED for d not in {64, 128} or k > 4096,
 * RT_ERR_WORKSPACE for a missing or short workspace (as rt_centroid_ema). */
rt_status rt_centroid_ema_topw(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                               const int32_t* idx, int w, float* centroids, int k, float decay,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Local (sliding-window) causal attention, the layer the pages pair with
 * routing attention (§3: causal and local attention choose each query's keys
 * from positions alone; §6 "Local vs Global": local attention with windows of
 * 512 and 1024 positions, combined with routing layers):
 *   out[b,h,t] = sum_{s = max(0, t-window+1)}^{t} softmax_s(scale <q_t, k_s>) v_s
 * (the window counts the position itself: window 1 returns V).
 *   q, k, v  [B,H,n,d] bf16 (dt must be RT_BF16; RT_F32 -> RT_ERR_UNSUPPORTED);
 *            shared QK only: k must be the same pointer as q
 *   window   >= 1 (a window >= n is full causal attention)
 *   scale    <= 0 selects 1/sqrt(d)
 *   out      [B,H,n,d] bf16 (fp32 accumulation, one rounding)
 *   workspace at least 256 bytes, 256-byte aligned (its first word is the
 *            device status word, as for the other calls)
 * d in {64, 128}; tcgen05 tensor cores, 128-row query tiles walking their
 * window's 128-position key blocks with an online softmax. */
rt_status rt_local_attention(const void* q, const void* k, const void* v, rt_dtype dt,
                             int B, int H, int n, int d, int window, float scale, void* out,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Clears the device status word at the start of a new workspace (an async
 * memset of its first 256 bytes on `stream`).  Call once after allocating a
 * workspace; the compute calls only ever set the word. */
rt_status rt_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Routing for callers that cannot allocate device memory.  The paper has no
 * counterpart to this call: it exists for callers that cannot call cudaMalloc
 * (or any allocating routine) where they route -- code running inside a host
 * framework whose device allocator it does not own, or a program that fixes
 * its device footprint at start-up -- and so cannot provide the workspace
 * rt_route_assign needs for its score matrix.
 *
 * Same computation and outputs as rt_route_assign (no `scores` output), with
 * the fp32 score scratch [B,H,k,n] taken from a fixed array in device memory
 * that the library owns: at most RT_NOALLOC_MAX_SCORES elements (32 MiB),
 * held on every GPU that loads the library until the process exits.  Larger
 * B*H*k*n returns RT_ERR_UNSUPPORTED before anything is launched.
 *   - allocates nothing: no cudaMalloc/cudaFree, no allocating library call;
 *   - the first call on a device (with that device current) looks up the
 *     array's device address once; make that first call before any stream
 *     capture;
 *   - every call shares the one array, so calls that overlap on the GPU
 *     (other streams, other host threads) race; serialise them.
 *   qk [B,H,n,d] dtype dt, centroids [H,k,d] fp32, idx [B,H,k,w] out,
 *   assign [B,H,n] out or NULL, stream as elsewhere. */
#define RT_NOALLOC_MAX_SCORES (8u * 1024u * 1024u)
rt_status rt_route_assign_noalloc(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                                  const float* centroids, int k, int w,
                                  int32_t* idx, int32_t* assign, void* stream);

/* Synchronises `stream`, reads the device error word kept in `workspace`,
 * clears it, and returns RT_OK, RT_ERR_TIMEOUT or RT_ERR_CUDA.  Not for use
 * inside stream capture. */
rt_status rt_check_device_status(void* workspace, size_t workspace_bytes, void* stream);

/* Human-readable name of a status code (static string). */
const char* rt_status_string(rt_status s);

/* Detail of the last error returned on the calling host thread (static
 * thread-local buffer; empty string if none). */
const char* rt_last_error_detail(void);

/* Number of kernels this library has launched since it was loaded (all
 * threads).  Used by benchmarks to count launches in a timed region. */
int64_t rt_launch_count(void);

/* Per-launch timing hook for benchmarks.  While set, the i-th kernel the
 * library launches after this call (i < n_pairs) records events[2i] just
 * before and events[2i+1] just after itself on its stream.  `events` are
 * cudaEvent_t handles created by the caller with timing enabled; the array
 * is copied.  rt_profile_set(NULL, 0) switches the hook off. */
rt_status rt_profile_set(void* const* events, int n_pairs);

/* Kernel-kind id of the i-th launch recorded since rt_profile_set (or -1),
 * and the name of a kernel kind. */
int rt_profile_kernel_id(int i);
const char* rt_kernel_name(int id);

#ifdef __cplusplus
}
#endif

#endif /* ROUTING_ATTENTION_H */
