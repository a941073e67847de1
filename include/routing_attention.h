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
 *     workspace and reported by rt_check_device_status(), which clears it;
 *     the outputs of the call that failed are undefined (the later kernels
 *     of that call still run, and every index they follow is bounds-checked,
 *     so no access leaves its buffer).
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
 *   q, k, v   [B,H,n,d]  dtype dt; shared QK when k is the same pointer as q;
 *                        a different k routes the keys separately (see
 *                        rt_routing_attention_separate; idx_out then holds
 *                        the queries' lists)
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

/* One training step of the layer: the forward pass of rt_routing_attention
 * (shared QK) followed by the centroid step of rt_centroid_ema on the same
 * rows and the assignment the forward computed -- the routing uses the
 * centroids as they were, then they move.  Source: §4 "Routing attention with
 * clustering" (centroids learned online while the layer runs), §2.
 * The centroid step needs only the assignment, so it runs on a second stream
 * the library owns (one per device, created by the first call; make that
 * call before any stream capture), forked from `stream` once the assignment
 * exists and joined back before the call's last operation: the caller sees
 * one stream, and the step captures into a CUDA graph as a fork and a join.
 * Calls from several host threads are serialised around the fork.
 *   q, v        [B,H,n,d] dtype dt (queries double as keys)
 *   centroids   [H,kc,d] fp32, read by the routing, then updated in place
 *   decay       in [0, 1]
 *   out, idx_out, assign_out, causal, scale: as rt_routing_attention
 *   workspace   rt_workspace_bytes(B, H, n, d, kc, w, dt) bytes
 * Results equal rt_routing_attention followed by rt_centroid_ema. */
rt_status rt_routing_attention_step(const void* q, const void* v, rt_dtype dt, int B, int H,
                                    int n, int d, float* centroids, int kc, int w, int causal,
                                    float scale, float decay, void* out, int32_t* idx_out,
                                    int32_t* assign_out, void* workspace, size_t workspace_bytes,
                                    void* stream);

/* Routing attention with separate queries and keys.
 * Source: §4 "Routing attention with clustering" (queries and keys are
 * routed to the same learned centroids; a query attends only to the keys of
 * its own clusters), §3 (softmax attention, causal masking).  Read as: the
 * queries and the keys are each normalised and scored against the centroids,
 * and every centroid keeps its w best queries and, separately, its w best
 * keys (ascending positions, ties to the lower position).  In cluster c each
 * listed query attends with softmax to the cluster's listed keys (with
 * causal=1 only to keys at positions not after its own).  A position's output
 * is the mean over the clusters that listed it as a query AND gave it at
 * least one visible key; a position with none gets a zero row.
 *   q, k, v    [B,H,n,d] dtype dt; k must be a different tensor from q
 *              (RT_ERR_INVALID_ARG otherwise; shared QK is
 *              rt_routing_attention)
 *   idx_q_out  [B,H,kc,w] out, may be NULL: the queries' lists
 *   idx_k_out  [B,H,kc,w] out, may be NULL: the keys' lists
 *   assign_out [B,H,n]    out, may be NULL: argmax centroid of every query
 *   the rest as for rt_routing_attention (same workspace size).
 * bf16: tcgen05 tensor cores (any w); fp32: CUDA cores. */
rt_status rt_routing_attention_separate(const void* q, const void* k, const void* v,
                                        rt_dtype dt, int B, int H, int n, int d,
                                        const float* centroids, int kc, int w,
                                        int causal, float scale, void* out,
                                        int32_t* idx_q_out, int32_t* idx_k_out,
                                        int32_t* assign_out, void* workspace,
                                        size_t workspace_bytes, void* stream);

/* Backward pass of rt_routing_attention (shared QK) with the routing held
 * fixed: the gradients of the loss with respect to the rows, given its
 * gradient with respect to `out`.
 * Source: §3 (softmax attention), §4 (attention only between same-cluster
 * pairs; centroids learned by the online k-means step, not by gradients --
 * §2).  The routing is piecewise constant in the rows, so the gradient flows
 * through the attention of each cluster and the averaging of a position's
 * cluster outputs: with m(t) the number of clusters listing t and, per
 * cluster, P = softmax(scale Q_c Q_c^T + causal mask), dY = dout[p]/m(p),
 *   dV_c = P^T dY;  dS = P * (dY V_c^T - rowsum(P * (dY V_c^T)));
 *   dQ_c = scale (dS Q_c + dS^T Q_c)   (a row is both a query and a key),
 * and each position's gradient is the sum of its rows over its clusters.
 *   q, v      [B,H,n,d] dtype dt (the forward's inputs; k was q)
 *   idx       [B,H,kc,w] int32: the forward's index lists (idx_out)
 *   causal, scale: as passed to the forward
 *   dout      [B,H,n,d] fp32: gradient with respect to out
 *   dq, dv    [B,H,n,d] fp32 out: gradients with respect to q (= k) and v;
 *             positions in no cluster get zero rows
 * The clusters are processed on CUDA cores in fp32 (P is recomputed), with
 * per-slot rows summed per position in ascending cluster order: the result is
 * deterministic.  Workspace: rt_workspace_bytes(B, H, n, d, kc, w, dt). */
rt_status rt_routing_attention_backward(const void* q, const void* v, rt_dtype dt, int B, int H,
                                        int n, int d, const int32_t* idx, int kc, int w,
                                        int causal, float scale, const float* dout, float* dq,
                                        float* dv, void* workspace, size_t workspace_bytes,
                                        void* stream);

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
 * A segmented reduction: the rows are first sorted by assigned centroid
 * chunk by chunk (integer counts only), then each centroid's rows are summed
 * in that fixed order, with no floating-point atomics: results are
 * deterministic.  Needs a workspace of at least
 * rt_workspace_bytes(B, H, n, d, k, 1, dt) bytes (row ids and per-chunk
 * counts live there). */
rt_status rt_centroid_ema(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                          const int32_t* assign, float* centroids, int k, float decay,
                          void* workspace, size_t workspace_bytes, void* stream);

/* The centroid step split for a batch sharded over several GPUs (one process
 * per GPU, each holding some of the sequences).  The step's means run over
 * every sequence of the batch (§4: centroids shared across sequences), so
 * each shard computes its own sums, the shards' sums are added with one
 * all-reduce (the caller's collective, e.g. NCCL), and every shard applies the
 * same blend:
 *   rt_centroid_ema_sums:  sums[h][c][0..d) = sum of r_t over this shard's
 *                          rows with assign == c; sums[h][c][d] = their count
 *                          (as a float, exact below 2^24);
 *   (all-reduce sums over the shards: elementwise addition)
 *   rt_centroid_ema_apply: for every (h, c) with count N > 0,
 *                          mu_c <- normalise(decay*mu_c + (1-decay)*sum/N);
 *                          other centroids are left bit-exact.
 * With one shard the two calls give rt_centroid_ema's result (the sums are
 * taken in the same fixed order).
 *   sums      [H,k,d+1] fp32 (written by _sums; read by _apply)
 *   the other arguments as for rt_centroid_ema; _sums needs the same
 *   workspace, _apply none. */
rt_status rt_centroid_ema_sums(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                               const int32_t* assign, int k, float* sums,
                               void* workspace, size_t workspace_bytes, void* stream);
rt_status rt_centroid_ema_apply(const float* sums, int H, int d, float* centroids, int k,
                                float decay, void* stream);

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

/* A layer with local heads and routing heads on the same tensors, as the
 * pages combine them (§6 "Local vs Global": local attention with windows of
 * 512 or 1024 positions in some heads, routing attention in others; §3, §4).
 * Heads [0, n_local) take causal local attention over `window` positions
 * (rt_local_attention); heads [n_local, H) take routing attention with
 * shared QK (rt_routing_attention, causal as given).  Within one sequence the
 * heads of each kind are contiguous in memory, so the call launches each kind
 * once per sequence on the caller's tensors (no copies).
 *   q, v        [B,H,n,d] dtype dt (local heads need bf16)
 *   centroids   [H - n_local, kc, d] fp32: the routing heads' centroids
 *   out         [B,H,n,d] dtype dt, every row written
 *   idx_out     [B, H - n_local, kc, w] out, may be NULL
 *   assign_out  [B, H - n_local, n] out, may be NULL (argmax per row; the
 *               centroid step of the routing heads: rt_centroid_ema_sums on
 *               each sequence's routing heads, added, then
 *               rt_centroid_ema_apply)
 *   workspace   at least rt_workspace_bytes(1, H - n_local, n, d, kc, w, dt)
 *               bytes (256 when every head is local)
 * Errors as the two calls it makes; both halves are checked before anything
 * is launched. */
rt_status rt_mixed_attention(const void* q, const void* v, rt_dtype dt, int B, int H, int n,
                             int d, int n_local, int window, const float* centroids, int kc,
                             int w, int causal, float scale, void* out, int32_t* idx_out,
                             int32_t* assign_out, void* workspace, size_t workspace_bytes,
                             void* stream);

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
 * that the library owns: at most RT_NOALLOC_MAX_SCORES elements (32 MiB) per
 * CUDA context that uses this call, held until the process exits.  Larger
 * B*H*k*n returns RT_ERR_UNSUPPORTED before anything is launched.
 *   - allocates nothing itself: no cudaMalloc/cudaFree, no allocating
 *     library call.  With lazy module loading (the CUDA default) the 32 MiB
 *     are reserved by the driver when the first call in a context looks up
 *     the array's address, so that first call may fail with RT_ERR_CUDA when
 *     device memory is short: callers with a fixed memory budget should make
 *     their first call at start-up;
 *   - the first call in each context (with that context's device current)
 *     looks the array's device address up once and caches it under the
 *     context's unique id; make that first call before any stream capture;
 *   - every call shares the one array, so calls that overlap on the GPU
 *     (other streams, other host threads) race; serialise them;
 *   - a device-side bounded wait that runs out is recorded in a status word
 *     the library also keeps per context; rt_check_device_status(NULL, 0,
 *     stream) reads and clears it.
 *   qk [B,H,n,d] dtype dt, centroids [H,k,d] fp32, idx [B,H,k,w] out,
 *   assign [B,H,n] out or NULL, stream as elsewhere. */
#define RT_NOALLOC_MAX_SCORES (8u * 1024u * 1024u)
rt_status rt_route_assign_noalloc(const void* qk, rt_dtype dt, int B, int H, int n, int d,
                                  const float* centroids, int k, int w,
                                  int32_t* idx, int32_t* assign, void* stream);

/* Synchronises `stream`, reads the device error word kept in `workspace`,
 * clears it, and returns RT_OK, RT_ERR_TIMEOUT or RT_ERR_CUDA.  The word
 * stays set from the failure until this call, across later calls.  With
 * workspace == NULL and workspace_bytes == 0 it reads (and clears) the status
 * word of rt_route_assign_noalloc in the current context instead.  Not for
 * use inside stream capture. */
rt_status rt_check_device_status(void* workspace, size_t workspace_bytes, void* stream);

/* Test aid for the device-side timeout path; not for production use.  While
 * `kernels` is non-zero, every later launch of the selected kernels begins
 * with a wait, bounded by limit_ns (0 < limit_ns <= 1e9), on a barrier that
 * nothing arrives on -- before the kernel issues any asynchronous copy or
 * tensor-core operation -- so the wait runs out: the kernel sets the device
 * status word (RT_ERR_TIMEOUT from rt_check_device_status) and returns with
 * nothing in flight; the outputs of that call are undefined.
 * rt_debug_inject_wait_timeout(0, 0) turns it off.  Process-wide setting,
 * read when a kernel is launched.  RT_ERR_INVALID_ARG for unknown bits or a
 * limit outside the range. */
#define RT_DEBUG_SCORE 1u            /* the tensor-core score kernel            */
#define RT_DEBUG_ATTENTION 2u        /* the tensor-core cluster-attention kernels */
#define RT_DEBUG_LOCAL_ATTENTION 4u  /* the local-attention kernel               */
rt_status rt_debug_inject_wait_timeout(unsigned kernels, unsigned long long limit_ns);

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
 * is copied.  On a stream that is being captured into a CUDA graph the
 * events are recorded as external event nodes, so each replay records them.
 * rt_profile_set(NULL, 0) switches the hook off. */
rt_status rt_profile_set(void* const* events, int n_pairs);

/* Kernel-kind id of the i-th launch recorded since rt_profile_set (or -1),
 * and the name of a kernel kind. */
int rt_profile_kernel_id(int i);
const char* rt_kernel_name(int id);

#ifdef __cplusplus
}
#endif

#endif /* ROUTING_ATTENTION_H */
