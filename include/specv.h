/*
 * specv.h -- C ABI of the GB300 lossless draft-verification library.
 *
 * The library implements, as CUDA kernels for sm_103a, the data-parallel step
 * of lossless speculative decoding that sits between the target model's
 * forward pass and the commit of tokens:
 *
 *   specv_verify_chain        chain speculative sampling (accept / first
 *                             rejection / residual or bonus token) and, at
 *                             temperature 0, greedy argmax verification
 *   specv_verify_tree_greedy  greedy verification of a linearised candidate tree
 *   specv_dart_tree           DART's candidate tree (top-k per offset, beam, node budget)
 *   specv_markov_draft        the DSpark Markov draft head, sampled position by position
 *   specv_markov_recompute_logits  the draft logits of the verified positions, recomputed
 *   specv_tv_accept           the analytic acceptance c* = 1 - 1/2 ||p_d - p_t||_1
 *   specv_schedule            DSpark's greedy throughput scheduler
 *   specv_schedule_global     its asynchronous global-search form (dynamic top-K)
 *   specv_prune_threshold     confidence-threshold suffix pruning
 *   specv_confidence_head     DSpark's confidence head c_k over all draft positions
 *   specv_shard_*             host combines of per-shard partials for rows whose
 *                             vocabulary is split over several GPUs
 *
 * Sources (cited per entry point below):
 *   [DART notes]   "DART：把草稿并行生成之后，还要补上哪些依赖？", DART reading
 *                  notes, zhongzhuzhou.org, 2026-10-14.
 *   [DSpark guide] DSpark paper guide, personal-site-bgy.pages.dev/ai-notes/
 *                  dspark-paper-guide.html.
 *   [SD survey]    "投机解码综述", zhifeiding.github.io, 2026-11-02.
 *
 * Notation: q = target distribution, p = draft distribution (DART notes §2.3).
 * q = softmax(target_logits / T), p = softmax(draft_logits / T); T = 0 selects
 * greedy (argmax) verification.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every array pointer is a caller-owned DEVICE pointer on the current CUDA
 *    device, row-major and contiguous, aligned at least to its element size.
 *    The library never allocates, frees or keeps pointers after a call returns.
 *  - Scratch memory: each entry point takes a caller-owned device `workspace`
 *    of at least specv_*_workspace_size(...) bytes, 256-byte aligned.  Its
 *    first 256 bytes hold the device error word (see specv_read_device_error);
 *    the rest needs no initialisation.  Two calls that may run concurrently
 *    must not share a workspace.
 *  - All work is enqueued on `stream` (a cudaStream_t passed as void*; NULL =
 *    the legacy default stream).  No call synchronises; outputs are valid when
 *    the stream reaches the point after the call.  Calls allocate nothing and
 *    can be enqueued repeatedly with the same arguments.
 *  - Host-side validation happens before anything is enqueued: a bad argument
 *    returns SPECV_ERR_INVALID_ARG (or SPECV_ERR_UNSUPPORTED for a valid but
 *    unsupported shape/device) and nothing is launched.  A launch failure
 *    returns SPECV_ERR_CUDA.
 *  - Bad data that only the device can see (a token id outside [0, V), a
 *    uniform outside [0, 1), a malformed tree) never traps: the affected
 *    request's outputs are set to -1 and the device error word records
 *    SPECV_ERR_DEVICE_DATA; read it with specv_read_device_error.
 *  - Logits may be float32 or bfloat16 (SPECV_F32 / SPECV_BF16).  All
 *    arithmetic is float32; argmax compares the stored values exactly and
 *    resolves ties to the lowest token id.  Logits must be finite.
 *  - Thread-safe: no global state other than a per-device capability cache
 *    and the built-in scratch of specv_verify_chain_noalloc.  The one
 *    exception: specv_verify_chain_noalloc calls on one device share that
 *    scratch, so they must be serialised (see its section).
 */
#ifndef SPECV_H_
#define SPECV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SPECV_API __attribute__((visibility("default")))
#else
#define SPECV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define SPECV_ABI_VERSION 1
#define SPECV_MAX_GAMMA 32          /* draft positions per request (chain)        */
#define SPECV_MAX_TREE_NODES 1024   /* nodes per tree including the root          */
#define SPECV_MAX_TREE_DEPTH 64
#define SPECV_MAX_SCHED_ENTRIES 8192 /* R * gamma for specv_schedule              */
#define SPECV_MAX_MARKOV_RANK 1024
#define SPECV_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20) /* specv_verify_chain_noalloc */

typedef enum {
  SPECV_OK = 0,
  SPECV_ERR_INVALID_ARG = 1,   /* a host-visible argument is invalid; nothing enqueued */
  SPECV_ERR_UNSUPPORTED = 2,   /* valid request the build cannot serve (device, size)   */
  SPECV_ERR_CUDA = 3,          /* a CUDA call or launch failed                          */
  SPECV_ERR_DEVICE_DATA = 4,   /* device-detected bad data (outputs of that request = -1) */
  SPECV_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up                    */
  SPECV_ERR_SCRATCH_LIMIT = 6  /* shape needs more than specv_verify_chain_noalloc's
                                  built-in scratch (SPECV_NOALLOC_SCRATCH_BYTES)        */
} specv_status;

typedef enum { SPECV_F32 = 0, SPECV_BF16 = 1 } specv_dtype;

/* ------------------------------------------------------------------ chain */

/*
 * specv_verify_chain -- chain speculative sampling over full-vocabulary logits.
 *
 * Follows [DART notes] §2.3 eq. (3)-(4), [DSpark guide] (verification rule,
 * prefix survival, bonus token) and [SD survey] §1.2-§1.3.  For each request r
 * with draft length l_r (lengths[r], or gamma when lengths == NULL):
 *   for k = 0 .. l_r-1, left to right: accept x_k iff
 *       uniforms[r,k,0] < min(1, q_k(x_k) / p_k(x_k))       (p_k(x_k) = 0 accepts)
 *   the first rejection at k stops the chain: accepted_len[r] = k and
 *       out_token[r] is drawn from the residual r(v) = [q_k(v) - p_k(v)]_+ / R
 *       with the uniform uniforms[r,k,1] (R = sum_v [q_k - p_k]_+; if R == 0
 *       the draw is from q_k);
 *   with no rejection accepted_len[r] = l_r and out_token[r] is the bonus token
 *       drawn from q_{l_r} with uniforms[r,l_r,1].
 *   A draw from weights w uses the inverse CDF over ascending token id:
 *       y = min{ v : sum_{v' <= v} w(v') > u * sum_v w(v) }.
 * The committed tokens of request r are x_0 .. x_{A-1} followed by out_token[r]
 * (A + 1 tokens).
 *
 * T == 0: greedy verification ([SD survey] §1.3): g_k = argmax target[r,k,:];
 *   accepted_len = first k < l_r with x_k != g_k (else l_r); out_token = g_A.
 *   `uniforms` is not read and may be NULL.
 *
 * c_star (optional, may be NULL): c*_{r,k} = 1 - 1/2 ||p_k - q_k||_1 for
 *   k < l_r ([DSpark guide], analytic acceptance); NaN for k >= l_r.  At T = 0
 *   it is 1 when argmax draft_k == argmax target_k, else 0.
 *
 * Arguments
 *   target_logits  [R, gamma+1, V]  dtype   row (r,k) = target logits that verify x_k;
 *                                            row (r,l_r) is the bonus row
 *   draft_logits   [R, gamma, V]    dtype   may be NULL only if T == 0 and c_star == NULL
 *   draft_tokens   [R, gamma]       int32   x_{r,k} in [0, V)
 *   lengths        [R] int32 or NULL        0 <= l_r <= gamma
 *   uniforms       [R, gamma+1, 2]  float32 in [0, 1); [.,.,0] accept test,
 *                                            [.,.,1] residual/bonus draw
 *   R >= 0, 0 <= gamma <= SPECV_MAX_GAMMA, V >= 1, temperature >= 0 (finite)
 *   accepted_len   [R] int32 out    A_r, or -1 on device-detected bad data
 *   out_token      [R] int32 out    correction or bonus token, or -1
 *   c_star         [R, gamma] float32 out, or NULL
 * Errors: SPECV_ERR_INVALID_ARG for NULL/negative/misaligned arguments or a
 *   workspace that is too small; SPECV_ERR_UNSUPPORTED if V is beyond what the
 *   kernels tile (specv_verify_chain_workspace_size returns 0 then).
 */
SPECV_API size_t specv_verify_chain_workspace_size(int R, int gamma, int V, specv_dtype dtype);
SPECV_API specv_status specv_verify_chain(const void* target_logits, const void* draft_logits, specv_dtype dtype,
                                const int32_t* draft_tokens, const int32_t* lengths, const float* uniforms,
                                int R, int gamma, int V, float temperature,
                                int32_t* accepted_len, int32_t* out_token, float* c_star,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * specv_verify_chain_noalloc -- specv_verify_chain without a caller workspace.
 *
 * The pages have no counterpart: this is a library convenience.  It computes
 * exactly what specv_verify_chain computes, with the same kernels and
 * arguments minus (workspace, workspace_bytes).  The scratch is a static
 * device buffer of SPECV_NOALLOC_SCRATCH_BYTES (16 MiB) per device, built into
 * the library, so the call allocates and frees nothing.  It serves callers
 * that cannot hand over device memory: code running inside an allocator or
 * memory-pool callback, servers that forbid device allocation once their
 * weights and KV cache are placed, C hosts without a device allocator.
 *
 * Set-up: the first call on each device (with that device current) loads
 *   the library's device module there through cudaGetSymbolAddress; make that
 *   first call outside any stream capture.  Every call looks the buffer's
 *   address up again (a host-side lookup once the module is loaded), so the
 *   address stays right after cudaDeviceReset and in any context the caller
 *   makes current.
 * Concurrency: all calls on one device share the one buffer.  Calls whose
 *   execution may overlap (different streams, or host threads enqueueing
 *   without ordering) race on it and give undefined results; serialise them
 *   on one stream.
 * Device-detected bad data still gives -1 outputs for the request; the error
 *   word itself stays inside the built-in buffer and is not readable.
 * Errors: as specv_verify_chain; SPECV_ERR_INVALID_ARG also when
 *   specv_verify_chain_workspace_size(R, gamma, V, dtype) is 0, and
 *   SPECV_ERR_SCRATCH_LIMIT when it exceeds SPECV_NOALLOC_SCRATCH_BYTES
 *   (e.g. R = 1024, gamma = 7, V = 151936 bf16 needs about 8.1 MiB and fits;
 *   R = 2048 needs 16.25 MiB and does not).  Both are decided on the host before any CUDA call.
 */
SPECV_API specv_status specv_verify_chain_noalloc(const void* target_logits, const void* draft_logits,
                                       specv_dtype dtype, const int32_t* draft_tokens, const int32_t* lengths,
                                       const float* uniforms, int R, int gamma, int V, float temperature,
                                       int32_t* accepted_len, int32_t* out_token, float* c_star, void* stream);

/* ------------------------------------------------------------------ c* */

/*
 * specv_tv_accept -- analytic acceptance c*_{r,k} = 1 - 1/2 ||p_k - q_k||_1
 * ([DSpark guide], the confidence head's supervision target; equal to
 * sum_v min(p_k, q_k) = 1 - R by [DART notes] eq. (3)).
 *   target_logits  [R, target_positions, V] dtype, rows k < gamma are used
 *   draft_logits   [R, gamma, V] dtype
 *   target_positions >= gamma (e.g. gamma + 1 when the bonus row is present)
 *   c_star         [R, gamma] float32 out.  At T = 0: argmax agreement (1 or 0).
 */
SPECV_API size_t specv_tv_accept_workspace_size(int R, int gamma, int V, specv_dtype dtype);
SPECV_API specv_status specv_tv_accept(const void* target_logits, const void* draft_logits, specv_dtype dtype,
                             int R, int gamma, int target_positions, int V, float temperature,
                             float* c_star, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------ tree */

/*
 * specv_verify_tree_greedy -- greedy (T = 0) verification of a linearised
 * candidate tree ([DART notes] §2.3 last paragraph and Algorithm 3 steps 9-10;
 * [SD survey] §2.3).
 *   Node 0 is the root (the committed prefix); node i >= 1 carries token
 *   tokens[r,i] and has parent parents[r,i] with 0 <= parents[r,i] < i
 *   (ancestors precede descendants).  Row i of target_logits is the target's
 *   distribution after node i.  g_i = argmax row i (lowest id on ties).
 *   Node i is accepted iff its parent is accepted and tokens[r,i] == g_{parent}.
 *   i* = accepted node of greatest depth (lowest index on ties).
 *   path_len[r] = depth of i*, path_nodes[r,:] = the nodes root->i* without the
 *   root (-1 padded), out_token[r] = g_{i*} (correction / bonus token).
 *   target_logits [R, N+1, V] dtype; parents, tokens [R, N+1] int32
 *   (parents[r,0] = -1, tokens[r,0] ignored); 1 <= max_depth <= SPECV_MAX_TREE_DEPTH;
 *   0 <= N, N+1 <= SPECV_MAX_TREE_NODES.
 *   path_len [R], path_nodes [R, max_depth], out_token [R] int32 out.
 *   A malformed tree (bad parent, depth > max_depth, token outside [0, V))
 *   gives -1 outputs for that request and SPECV_ERR_DEVICE_DATA.
 */
SPECV_API size_t specv_verify_tree_greedy_workspace_size(int R, int N, int V, specv_dtype dtype);
SPECV_API specv_status specv_verify_tree_greedy(const void* target_logits, specv_dtype dtype,
                                      const int32_t* parents, const int32_t* tokens,
                                      int R, int N, int V, int max_depth,
                                      int32_t* path_len, int32_t* path_nodes, int32_t* out_token,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------ candidate tree */

/*
 * specv_dart_tree -- DART's candidate-tree construction without the n-gram
 * index [DART notes §5.2-5.3 and Algorithm 3 steps 1-8, with the n-gram score
 * g == 1]: for future offsets i = 1..d, K_i = the top-k tokens of
 * p_i = softmax(draft_logits[:, i-1] / T) (lower id first on equal logits);
 * starting from the root (score 0) every active path is extended by every token
 * of K_i with eq. (10)'s increment
 *   (0.9^i ln(p_i(v) + eps) + 0.5 ln(1 + eps)) / (i + 1)^0.7,   eps = 1e-10,
 * all extensions join the node set T (at most k + (d-1) w k nodes, eq. (9)) and
 * the w best (score, then generation order) stay active.  The theta nodes of T
 * with the largest key = min(score, parent's key) (then smaller depth, then
 * generation order) form the tree, which is ancestor-closed by construction.
 * Output, ready for specv_verify_tree_greedy: row 0 is the root (the committed
 * prefix, parents -1, token 0); rows 1 .. n_nodes-1 are the selected nodes in
 * depth-first preorder, children in selection order; parents[i] < i.
 *   draft_logits [R, d, V] dtype, 16-byte aligned rows (V a multiple of 8 for
 *     bf16, 4 for float32), at most 128 tiles of 2560 (bf16) / 1280 (float32)
 *     elements per row; T > 0.
 *   1 <= d <= 8, 1 <= k <= min(32, V), 1 <= w <= 32, 1 <= theta <= 1023; T's
 *     k + (d-1) w k nodes, 40 bytes each, must fit 200 KB of shared memory
 *     (the default (d, k, w, theta) = (8, 25, 20, 59) uses 138 KB).
 *   parents, tokens [R, theta + 1] int32 out (rows past n_nodes: -1 and 0);
 *   n_nodes [R] int32 out (= min(theta, |T|) + 1).
 *   Workspace: specv_dart_tree_workspace_size bytes (0 means unsupported).
 * Errors: SPECV_ERR_INVALID_ARG for arguments outside these ranges, T <= 0 or
 *   a short workspace; SPECV_ERR_UNSUPPORTED for unaligned rows or a shape over
 *   the tile / shared-memory limits.
 */
SPECV_API size_t specv_dart_tree_workspace_size(int R, int d, int V, int k, int w, int theta, specv_dtype dtype);
SPECV_API specv_status specv_dart_tree(const void* draft_logits, specv_dtype dtype, int R, int d, int V,
                                       float temperature, int k, int w, int theta, int32_t* parents,
                                       int32_t* tokens, int32_t* n_nodes, void* workspace,
                                       size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------ Markov head */

/*
 * specv_markov_draft -- semi-autoregressive drafting with the DSpark Markov head
 * ([DSpark guide]: p_k(v | x_0, x_<k) = softmax(U_k(v) + B(x_{k-1}, v)),
 * B = W1 W2, W1 [V, rank] used as a row lookup, W2 [rank, V] as the projection).
 *   x_0 = anchor[r].  For k = 1 .. gamma (sequentially):
 *     L_k = U[r,k-1,:] + W1[x_{k-1},:] . W2            (float32 accumulation)
 *     x_k = inverse-CDF draw from softmax(L_k / T) with uniforms[r,k-1]
 *           (T = 0: argmax, lowest id on ties)
 *   U [R, gamma, V] bf16, W1 [V, rank] bf16, W2 [rank, V] bf16,
 *   anchor [R] int32, uniforms [R, gamma] float32 (may be NULL at T = 0).
 *   draft_tokens [R, gamma] int32 out (x_1 .. x_gamma).
 *   draft_logits [R, gamma, V] out or NULL: the raw L_k (before temperature)
 *   in logits_out_dtype (SPECV_F32 or SPECV_BF16).  The draw uses L_k in that
 *   precision (SPECV_BF16: rounded to bfloat16), also when draft_logits is
 *   NULL; then no logits are written at all (tensor-core form) and
 *   specv_markov_recompute_logits can later produce the rows a verification
 *   reads, equal to the ones drawn from.
 *   1 <= rank <= SPECV_MAX_MARKOV_RANK, rank % 16 == 0; V <= 262144 (larger V
 *   returns SPECV_ERR_UNSUPPORTED).
 * Execution: when rank is a multiple of 64 and at most 256, V is a multiple of
 *   8 and U, W1, W2 and draft_logits are 16-byte aligned, the contraction
 *   runs on the tensor cores (tcgen05, bf16 x bf16 -> float32, W2 read in
 *   place); other shapes use a CUDA-core kernel.
 *   Both accumulate the rank products in float32 (order unspecified).
 * Errors: SPECV_ERR_INVALID_ARG for bad sizes, NULL or misaligned pointers or
 *   a short workspace; a previous token outside [0, V) or a uniform outside
 *   [0, 1) gives draft token -1 and SPECV_ERR_DEVICE_DATA in the error word.
 */
SPECV_API size_t specv_markov_draft_workspace_size(int R, int gamma, int V, int rank);
SPECV_API specv_status specv_markov_draft(const void* U, const void* W1, const void* W2,
                                const int32_t* anchor, const float* uniforms,
                                int R, int gamma, int V, int rank, float temperature,
                                int32_t* draft_tokens, void* draft_logits, specv_dtype logits_out_dtype,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * specv_markov_recompute_logits -- the draft logits a chain verification
 * reads, recomputed after drafting without kept logits ([DSpark guide],
 * Markov head: L_k = U_k + W1[x_{k-1}] . W2; the verification rule reads
 * p_k only at the positions that are verified).
 *   For every request r and k < lengths[r] (all k < gamma when lengths is
 *   NULL): draft_logits[r, k, :] = L (bf16), with x_{k-1} = anchor[r] for
 *   k = 0 and draft_tokens[r, k-1] otherwise.  The sums run on the tensor
 *   cores with the tiling and summation order of specv_markov_draft's
 *   kept-logits form, so the rows are bitwise the bf16 logits a drafting call
 *   that keeps them writes; a drafting call that keeps none draws the same
 *   tokens as one that keeps them except at numerical near-ties of its CDF.
 *   Other rows of draft_logits are not written.
 *   U [R, gamma, V], W1 [V, rank], W2 [rank, V] bf16; anchor [R],
 *   draft_tokens [R, gamma], lengths [R] int32 (0 <= lengths[r] <= gamma);
 *   draft_logits [R, gamma, V] bf16 out.  Workspace of at least
 *   specv_markov_recompute_logits_workspace_size(R, gamma) bytes.
 * Shapes: rank a multiple of 64 and at most 256, V a multiple of 8, U, W1, W2
 *   and draft_logits 16-byte aligned; other shapes give SPECV_ERR_UNSUPPORTED.
 * Errors: SPECV_ERR_INVALID_ARG for bad sizes or pointers; a length outside
 *   [0, gamma] counts as 0 and sets SPECV_ERR_DEVICE_DATA; a previous token
 *   outside [0, V) gives that row W1 = 0.
 */
SPECV_API size_t specv_markov_recompute_logits_workspace_size(int R, int gamma);
SPECV_API specv_status specv_markov_recompute_logits(const void* U, const void* W1, const void* W2,
                                                     const int32_t* anchor, const int32_t* draft_tokens,
                                                     const int32_t* lengths, int R, int gamma, int V, int rank,
                                                     void* draft_logits, void* workspace, size_t workspace_bytes,
                                                     void* stream);

/* ------------------------------------------------------------------ scheduler */

/*
 * specv_schedule -- DSpark's greedy throughput scheduler ([DSpark guide],
 * scheduler section).  a_{r,j} = prod_{i<=j} c_{r,i} (float64, left to right);
 * B = sum_r (1 + l_r); tau = sum_r (1 + sum_{j<=l_r} a_{r,j}); Theta = tau * SPS(B).
 * All (r, j) form one pool sorted by a descending (ties: lower r, then lower j);
 * entries are taken from the top while Theta rises; the first entry with
 * Theta <= Theta_best (or B > B_max) stops the loop (early stop).
 * tau is accumulated in fixed point with quantum 2^-48 (a truncated), so the
 * result is exact and independent of summation order.
 *   conf  [R, gamma] float32 in [0, 1]; sps [B_max] float64, sps[B-1] = SPS(B) > 0;
 *   R <= B_max; R * gamma <= SPECV_MAX_SCHED_ENTRIES.
 *   lengths [R] int32 out; theta_best [1] float64 out or NULL (tau in tokens x SPS).
 *   A confidence outside [0, 1] (or NaN) gives lengths = -1 and SPECV_ERR_DEVICE_DATA.
 */
SPECV_API size_t specv_schedule_workspace_size(int R, int gamma);
SPECV_API specv_status specv_schedule(const float* conf, const double* sps, int R, int gamma, int B_max,
                            int32_t* lengths, double* theta_best,
                            void* workspace, size_t workspace_bytes, void* stream);

/* specv_schedule_global -- the scheduler's asynchronous form [DSpark guide,
 * production deployment: the batch size of the next step must be known before
 * the current step ends, so the truncation count K is computed from confidence
 * outputs two steps old, which isolates the decision from the tokens being
 * verified; with that causal barrier the early stop is removed and K comes
 * from an unconstrained global search, while the entries taken are the top K
 * of the pool ordered by the current cumulative confidences].
 *   K = argmax over n = 0 .. min(R * gamma, B_max - R) of
 *       Theta_n = tau_n * SPS(R + n), tau_n and Theta_n as in specv_schedule but
 *       on the pool built from conf_stale; the smallest n among equal Theta_n
 *       (n = 0, bonus positions only, is a candidate).
 *   lengths: the per-request counts among the top K entries of the pool built
 *       from conf (a_{r,j} descending, ties by (r, j)); theta_best = Theta_K of
 *       the stale pool, in tokens x SPS.
 *   conf, conf_stale [R, gamma] float32 in [0, 1]; conf_stale may be NULL or
 *   equal to conf (K and the entries then come from one pool).  Other
 *   arguments, the workspace (specv_schedule_workspace_size) and errors as for
 *   specv_schedule; a bad value in either confidence array gives -1 lengths.
 */
SPECV_API specv_status specv_schedule_global(const float* conf, const float* conf_stale, const double* sps,
                                             int R, int gamma, int B_max, int32_t* lengths, double* theta_best,
                                             void* workspace, size_t workspace_bytes, void* stream);

/* specv_confidence_head -- DSpark's confidence head [DSpark guide, confidence
 * head: for each draft position k a light linear projection plus a sigmoid over
 * the backbone hidden state h_k and the Markov embedding W1[x_{k-1}] outputs
 * c_k, the probability that position k passes verification given that all
 * earlier positions did; the scheduler multiplies them into a_{r,j}].
 *   c[r, k] = sigmoid(w[0:H] . h[r, k] + w[H:H+rank] . W1[x_{r,k-1}] + b),
 *   x_{r,0} = anchor[r], x_{r,k-1} = draft_tokens[r, k-2] for k >= 2 (the last
 *   draft token is not used).  Accumulated in float32.
 *   h [R, gamma, H] bf16; W1 [V, rank] bf16 (the Markov head's table);
 *   w [H + rank] float32; b finite; anchor [R], draft_tokens [R, gamma] int32;
 *   conf [R, gamma] float32 out.  16-byte aligned rows with H and rank multiples
 *   of 8 take the vector path; other shapes run element by element.
 *   Workspace: specv_confidence_head_workspace_size bytes (the error word).
 *   A token outside [0, V) gives NaN for that position and SPECV_ERR_DEVICE_DATA.
 */
SPECV_API size_t specv_confidence_head_workspace_size(int R, int gamma);
SPECV_API specv_status specv_confidence_head(const void* h, const void* W1, const float* w, float b,
                                             const int32_t* anchor, const int32_t* draft_tokens, int R, int gamma,
                                             int H, int V, int rank, float* conf, void* workspace,
                                             size_t workspace_bytes, void* stream);

/* specv_prune_threshold -- confidence-threshold suffix pruning [SD survey
 * §6.1: the confidence head's prefix survival s_i = prod_{j<=i} a_j; the
 * low-confidence suffix below a threshold is cut before verification, falling
 * back to a shorter draft].
 *   s_{r,i} = prod_{j<=i} conf[r, j] in float64, multiplied left to right;
 *   lengths[r] = the number of leading positions with s_{r,i} >= threshold
 *   (s does not increase, so the kept positions are a prefix).
 *   conf [R, gamma] float32 in [0, 1]; lengths [R] int32 out; threshold finite
 *   or +-inf (NaN is SPECV_ERR_INVALID_ARG).  Workspace: the
 *   specv_schedule_workspace_size bytes (the error word).  A confidence outside
 *   [0, 1] gives that request -1 and SPECV_ERR_DEVICE_DATA.
 */
SPECV_API specv_status specv_prune_threshold(const float* conf, int R, int gamma, double threshold,
                                             int32_t* lengths, void* workspace, size_t workspace_bytes,
                                             void* stream);

/* ------------------------------------------------------ vocabulary-sharded combine
 *
 * Host functions (no device work, no CUDA call) for rows whose V logits are
 * split over several GPUs in contiguous ascending slices, shard s holding
 * token ids [off_s, off_s + V_s), off_0 = 0.  Each GPU reduces its own slice;
 * the caller's communication layer gathers the per-shard partials (all
 * arrays below are shard-major: element (s, r) at s * rows + r); these
 * functions combine them identically on every rank.  Sums over shards
 * (sum_v min(q, p), the residual mass sum_v [q - p]_+) need no function: they
 * are plain all-reduce sums.  Arrays are caller-owned HOST memory.
 *
 * specv_shard_combine_normalisers -- softmax normaliser of a full row from
 * per-shard (max, sum of exponentials) pairs [DART notes §2.3: q and p are
 * softmaxes over the whole vocabulary].  Ex2 domain, as the kernels keep it:
 *   part [shards, rows, 2] float32: (m_c2, Z) = (max_v x_v * c2,
 *        sum_v 2^(x_v * c2 - m_c2)) over the shard's slice, c2 = log2(e)/T;
 *        a shard with no element (or all -inf) gives Z = 0 (m_c2 ignored).
 *   out  [rows, 2] float32: (M_c2, Z) with M_c2 = max over shards with Z > 0
 *        and Z = sum_s Z_s * 2^(m_c2,s - M_c2) (accumulated in float64, shards
 *        in ascending order); a row with no mass gives (-inf, 0).
 *
 * specv_shard_pick -- the shard an inverse-CDF draw over ascending token ids
 * lands in [DART notes eq. (4) for the residual r = [q-p]_+/R; DSpark guide for
 * the bonus draw from q]: the draw is y = min{v : C(v) > u * S}, C the
 * cumulative weight and S the total.  With P_s the mass of the shards before s
 * (float64, ascending s), the owning shard is the first s with
 * P_s + mass_s > u * S, and that shard draws y from its own slice as
 * min{v : C_s(v) > target}, C_s cumulative within the slice.
 *   mass [shards, rows] float64 >= 0: each shard's total draw weight;
 *   u [rows] float32 in [0, 1);
 *   shard_out [rows] int32: the owning shard, or -1 when the row has no mass;
 *   target_out [rows] float64: u * S - P_s (>= 0), the threshold inside it.
 *   If rounding leaves no shard past u * S, the last shard with mass is taken
 *   (the same rule as the in-shard draw's last positive weight).
 *   A negative or non-finite mass, or u outside [0, 1), is SPECV_ERR_INVALID_ARG.
 *
 * specv_shard_argmax_combine -- greedy argmax of a full row from per-shard
 * (max value, token id) pairs [SD survey §1.3]: the larger value wins, equal
 * values go to the lower token id (the same tie rule as within a shard).
 *   val [shards, rows] float32, idx [shards, rows] int32 (global token ids);
 *   a shard with no element gives val = -inf, idx = INT32_MAX.
 *   out [rows] int32: the row's argmax, or -1 if every shard was empty.
 *
 * All three return SPECV_ERR_INVALID_ARG for shards < 1, rows < 0 or a NULL
 * array when rows > 0; otherwise SPECV_OK.
 */
SPECV_API specv_status specv_shard_combine_normalisers(const float* part, int shards, int rows, float* out);
SPECV_API specv_status specv_shard_pick(const double* mass, int shards, int rows, const float* u,
                                        int32_t* shard_out, double* target_out);
SPECV_API specv_status specv_shard_argmax_combine(const float* val, const int32_t* idx, int shards, int rows,
                                                  int32_t* out);

/* ------------------------------------------------------------------ utilities */

/* Waits for `stream`, copies the device error word of `workspace` into
 * *status_out (SPECV_OK or SPECV_ERR_DEVICE_DATA / SPECV_ERR_TIMEOUT) and
 * leaves it unchanged.  Each entry point clears the word when it starts. */
SPECV_API specv_status specv_read_device_error(const void* workspace, void* stream, int32_t* status_out);

SPECV_API const char* specv_status_string(specv_status status);
SPECV_API int specv_abi_version(void);

/*
 * specv_selftest_bounded_wait -- exercises the library's bounded device-side
 * wait (the pages have no counterpart: this is a failure-detection check).
 *
 * One thread initialises an mbarrier that expects one arrival and waits on
 * its first phase with the same poll-limited wait the Markov kernel uses for
 * its copies.  arrive == 0: nothing ever arrives, so after max_polls polls the
 * wait gives up and the kernel records SPECV_ERR_TIMEOUT in the workspace
 * error word and returns (no trap; the context stays usable).  arrive != 0:
 * the thread arrives first, the wait succeeds and the word stays SPECV_OK.
 *   max_polls in [1, 65536]; workspace >= 256 bytes, 256-byte aligned.
 * Errors: SPECV_ERR_INVALID_ARG for a bad argument, SPECV_ERR_UNSUPPORTED off
 * sm_103, SPECV_ERR_CUDA for a launch failure.  Read the outcome with
 * specv_read_device_error.
 */
SPECV_API specv_status specv_selftest_bounded_wait(uint32_t max_polls, int arrive, void* workspace,
                                                   size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SPECV_H_ */
