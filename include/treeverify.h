/*
 * treeverify.h - C ABI of the tree-verification library (libtreeverify.so), sm_103a.
 *
 * One verification round of tree speculative decoding, on one GPU:
 *   tv_select_subtree   budgeted prefix-closed subtree from a block-marginal pool
 *   tv_select_subtree_adaptive  the same, cut where expected tokens per unit cost peak
 *   tv_tree_prep        ancestor bitmask, depth / position ids, child lists
 *   tv_tree_attention   tree-masked grouped-query attention over prefix KV + tree KV
 *   tv_verify_greedy    fused vocab pass + greedy longest-match walk + bonus token
 *   tv_verify_sample    fused vocab pass + min(1,p/q) walk + residual resampling
 *   tv_vocab_stats      the fused vocab pass alone (row argmax / lse, drafted-token p, q)
 *   tv_commit_accepted_kv  keep the accepted path's cache rows (contiguous), drop the rest
 *   tv_frontier_topw / tv_expand_children  one single-drafter tree-expansion step
 *   tv_prune_tree       per-parent child cap and depth-window re-rooting of a tree
 *
 * Conventions shared by every call
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless marked
 *     "host".  The library never allocates device memory: calls that need scratch take
 *     a caller-provided `workspace` of at least the size returned by the matching
 *     tv_*_workspace_size() query.  A workspace must be zero-filled once before its
 *     first use; every call leaves it ready for the next call (its counters return to
 *     zero).  Calls that share one workspace must not overlap on the GPU.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns a tv_status.  TV_OK means the work was enqueued; argument
 *     errors found on the host return a negative status and enqueue nothing.
 *   - Problems that only the device can see (a malformed parent array, an
 *     out-of-range token, a bounded wait that ran out) are OR-ed as TV_DEV_* bits into
 *     the caller's `*dev_status` word (a device int32 the caller zeroes and reads back).
 *     Outputs of an affected sequence are then unspecified but every kernel still
 *     terminates.  Nothing throws across this ABI.
 *   - Tree layout: per sequence b, `parent[b][0] = -1` (node 0 is the root = the last
 *     committed token) and 0 <= parent[b][i] < i for i >= 1.  N counts all nodes,
 *     root included.  Row u of a logits block is the target (or draft) distribution of
 *     the token that follows node u, so draft node c is judged with row parent[c].
 *   - Ragged batches (TAPS §4.1 stage 3: the selected subtree is large when the drafter
 *     is confident and small otherwise, so one call's sequences hold different node
 *     counts): rows after a sequence's last node hold parent -1 and are inactive
 *     padding, as tv_select_subtree* writes them past n_nodes.  Padding is trailing:
 *     sequence b's active rows are 0..n_b-1, n_b = the first row i >= 1 whose parent is
 *     -1 (or N); a row with parent >= 0 after a padding row sets TV_DEV_BAD_TREE.  Padding
 *     rows are no drafts: their tokens are not checked, they are nobody's children and
 *     get no output (each call below says what it leaves in their output rows).  Their
 *     logits and cache rows are still addressed as [B][N] blocks.
 *   - Logits / activations are row-major and contiguous.  bf16 is IEEE bfloat16.
 *   - The kernels of tv_select_subtree*, tv_tree_attention (tensor-core path) and
 *     tv_verify_* are launched with programmatic stream serialization: their CTAs may
 *     become resident while the previous kernel of the stream is still finishing, and
 *     each waits (griddepcontrol.wait) for that kernel to complete, with its memory
 *     visible, before it reads or writes any global memory.  Stream order and results
 *     are those of an ordinary launch; only the launch latency between dependent
 *     kernels is hidden (and the selection kernel lets its successor start early).
 *
 * Passages restated (the pages' titles):
 *   TAPS (Target-Aware Prefix-tree Selection for diffusion-drafted speculative
 *     decoding) §4.1-§4.2;  PTD (Progressive Tree Drafting) §3.1 tree construction;
 *   TreeGraft (adaptive multi-drafter grafting) §3.1 cumulative path score;
 *   "Speculative decoding principles" (blog): parallel verification, greedy
 *     acceptance, sampling acceptance alpha = min(1, p/q), residual (p-q)+ correction.
 */
#ifndef TREEVERIFY_H
#define TREEVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define TV_API __attribute__((visibility("default")))
#else
#define TV_API
#endif

typedef struct CUstream_st* tv_stream_t; /* identical to cudaStream_t */

typedef enum tv_dtype {
  TV_F32 = 0,  /* IEEE float32 */
  TV_BF16 = 1  /* bfloat16 (fp32 accumulation inside) */
} tv_dtype;

typedef enum tv_status {
  TV_OK = 0,
  TV_ERR_NULL = -1,        /* a required pointer is NULL */
  TV_ERR_SHAPE = -2,       /* a size is out of the supported range */
  TV_ERR_DTYPE = -3,       /* unknown or unsupported dtype for this call */
  TV_ERR_WORKSPACE = -4,   /* workspace missing or smaller than the query says */
  TV_ERR_ALIGN = -5,       /* a pointer or stride breaks an alignment rule */
  TV_ERR_UNSUPPORTED = -6, /* a combination the library does not implement */
  TV_ERR_CUDA = -7,        /* a CUDA runtime/driver call failed while enqueueing */
  TV_ERR_VALUE = -8        /* a scalar argument is out of range (temperature, scale) */
} tv_status;

/* Bits OR-ed into *dev_status by device code. */
#define TV_DEV_BAD_TREE 1   /* parent[] breaks parent[0] = -1, 0 <= parent[i] < i */
#define TV_DEV_BAD_TOKEN 2  /* a draft token is outside [0, V) or pool token invalid */
#define TV_DEV_TIMEOUT 4    /* a bounded wait inside a kernel ran out (pipeline stall) */

/* Human-readable name of a tv_status value (static string, never NULL). */
TV_API const char* tv_status_string(int status);

/* Library ABI version: (major << 16) | minor. */
TV_API int tv_version(void);

/* tv_philox4x32_10 - the counter-based generator that tv_verify_sample draws its
 * uniforms from: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers:
 * as easy as 1, 2, 3", SC'11), key = seed split into (low, high) 32-bit words.
 *   counters [n][4] uint32 (device), out [n][4] uint32 (device): the four output words of
 *   each counter.  The sampling walk's draw k of kind `kind` at node u of sequence b in
 *   round r uses counter (r mod 2^32, b, u, 2k + kind) and the uniform (x0 >> 8) * 2^-24.
 * Errors: n < 0 -> TV_ERR_SHAPE; NULL arrays with n > 0 -> TV_ERR_NULL; arrays not 16-byte
 * aligned -> TV_ERR_ALIGN.
 */
TV_API tv_status tv_philox4x32_10(uint64_t seed, const uint32_t* counters, int n, uint32_t* out,
                                  tv_stream_t stream);

/* tv_selftest_bounded_wait - exercise the failure path of the in-kernel bounded waits.
 * (No counterpart in the pages: it checks this library's own failure detection.)  One
 * warp waits on an mbarrier phase that nothing completes, through the same bounded wait
 * the attention and vocab pipelines use but with a limit of wait_us microseconds; the
 * wait gives up, the kernel ORs TV_DEV_TIMEOUT into *dev_status and returns, and the CUDA
 * context stays usable.  Nothing faults, traps or hangs.
 * Errors: dev_status NULL -> TV_ERR_NULL; wait_us outside 1..1000000 -> TV_ERR_VALUE.
 */
TV_API tv_status tv_selftest_bounded_wait(int wait_us, int32_t* dev_status, tv_stream_t stream);

/* ------------------------------------------------------------------------------------
 * tv_set_sm_partition - SM shares for running tv_tree_attention and tv_verify_* at the
 * same time on two streams.  The vocab pass then launches at most verify_sms CTAs (one
 * per SM) and the tensor-core attention plans its KV splits for attention_sms SMs, so
 * that the two grids can be resident together instead of queueing behind each other.
 * 0 (the default) means the whole device.  Process-wide, host-side; affects launches
 * made after the call.  Results do not depend on it beyond fp32 summation order.
 * Errors: a negative count -> TV_ERR_VALUE.
 */
TV_API tv_status tv_set_sm_partition(int verify_sms, int attention_sms);

/* ------------------------------------------------------------------------------------
 * tv_set_attention_variant - which tensor-core kernel tv_tree_attention uses for bf16.
 *   0  automatic (default): the variant (1 or 3) and KV split count that minimise a
 *      wave model of the run time (see tv_tree_attention_plan); paired tiles need
 *      G * N > 128
 *   1  one 128-row tile per CTA
 *   2  paired row tiles: one CTA streams the KV range once for two 128-row tiles
 *   3  paired row tiles with 64-key KV tiles and two S buffers per row tile, so S of
 *      the next KV tile is computed while the softmax of the current one runs; without
 *      KV splits and with a prefix of at least 64 N keys, the tile pairs of a KV head run
 *      as 2-CTA clusters that share each K/V tile (TMA multicast)
 *   4  variant 3's pipeline (in its earlier form with one S issuing thread for both row
 *      tiles) on a persistent grid of one CTA per SM (of the attention's
 *      share): the 64-key steps of all tile pairs are cut into equal contiguous ranges,
 *      one per CTA, so that the device stays busy when the tile pairs do not fill a
 *      whole number of waves; a tile pair cut between CTAs is merged through the
 *      workspace by the CTA that finishes its last piece.  Needs the workspace; shapes
 *      whose ranges would hold more than 8 pieces run variant 3.  Measured 3-6 %
 *      slower than that single-issuer variant 3 on the long-context shapes, which run
 *      at the GB300's power limit (more busy SMs lower the clock), so the automatic
 *      choice never takes it.
 *   5  variant 3 on SM pairs (tcgen05 cta_group::2): the two CTAs of a cluster hold the
 *      four row tiles of a KV head, and every S and PV product is one M = 256 MMA over
 *      a row tile of each, issued by the even CTA; each CTA loads half of every K tile
 *      (32 of its 64 keys) and of every V tile (64 of the 128 value columns).  D = 128
 *      only, without KV splits, where the tile pairs of a KV head come in twos; other
 *      shapes run variant 3.  Measured equal to variant 3 on the long-context shape
 *      (at a higher SM clock under the power limit) and 3-7 % slower on budget-sweep
 *      trees, so the automatic choice never takes it.
 * All compute the same result (up to fp32 summation order); the switch exists to
 * compare and test them.  Process-wide, host-side; affects launches made after the call.
 * Errors: a value outside 0..5 -> TV_ERR_VALUE.
 */
TV_API tv_status tv_set_attention_variant(int variant);

/* ------------------------------------------------------------------------------------
 * tv_set_attention_splits - KV splits of the tensor-core attention, for measurement and
 * tuning.  0 (default): chosen per launch from the device's cluster occupancy and the
 * KV length.  1..8: every (sequence, KV head, row tile group) is cut into that many KV
 * ranges (at most one per 128-key tile), merged inside one thread-block cluster.
 * Results do not depend on it beyond fp32 summation order.  Process-wide, host-side.
 * Errors: a value outside 0..8 -> TV_ERR_VALUE.
 */
TV_API tv_status tv_set_attention_splits(int splits);

/* ------------------------------------------------------------------------------------
 * tv_tree_prep - tree structure for the attention mask and position encoding.
 * PTD §3.1 "tree construction": node v observes pi(v) = {v} U pi(P(v)); its position
 * encoding follows |pi(v)|.
 *   parent     [B][N] int32
 *   depth      [B][N] int32 out: |pi(v)| - 1                              (may be NULL)
 *   pos        [B][N] int32 out: P + depth (0-based position ids)        (may be NULL)
 *   anc_mask   [B][N][W] uint32 out, W = ceil(N/32): bit (j%32) of word j/32 of row i
 *              is set iff j in pi(i)                                      (may be NULL)
 *   child_off  [B][N+1] int32 out, child_idx [B][N] int32 out: per sequence, the
 *              children of u are child_idx[child_off[u] .. child_off[u+1]) in
 *              ascending node index (child_idx[b][N-1] is unused)  (both or neither)
 * Padding rows (ragged batches): depth and pos -1, an all-zero mask row, no children;
 * child_idx holds -1 past the n_b - 1 edges and child_off[b][N] = n_b - 1.
 * Limits: 1 <= N <= 1024, B >= 1.  Launches one CTA per sequence.
 */
TV_API tv_status tv_tree_prep(const int32_t* parent, int B, int N, int P, int32_t* depth, int32_t* pos,
                       uint32_t* anc_mask, int32_t* child_off, int32_t* child_idx,
                       int32_t* dev_status, tv_stream_t stream);

/* ------------------------------------------------------------------------------------
 * tv_prune_tree - width and depth control of a draft tree.
 * PTD §3.1 "overhead constraints": every parent keeps at most max_children children,
 * the most confident ones (conf descending, ties to the lower index), and loses the
 * others with their subtrees; then, while the kept tree is more than depth_limit edges
 * deep, the root's lowest-index kept child becomes the root and everything outside its
 * subtree is pruned (the page's sliding-window stepping; nodes are numbered in the
 * order they were added).  Survivors are renumbered in their original order.
 *   parent [B][N] int32 (tree layout as above), conf [B][N] float (finite)
 *   old_to_new [B][N] out: new index of each node or -1
 *   new_parent [B][N] out: rows < n_kept[b] hold the new tree (-1 at its root), the
 *                 rest -1
 *   n_kept [B], new_root [B] out: count and the old index of the new root
 * Limits: 1 <= N <= 1024, max_children >= 1, depth_limit >= 1.  No workspace.
 */
TV_API tv_status tv_prune_tree(const int32_t* parent, const float* conf, int B, int N, int max_children,
                        int depth_limit, int32_t* old_to_new, int32_t* new_parent, int32_t* n_kept,
                        int32_t* new_root, int32_t* dev_status, tv_stream_t stream);

/* ------------------------------------------------------------------------------------
 * tv_tree_attention - tree-masked grouped-query attention of the draft tree.
 * PTD §3.1 (a node attends only to its ancestors), blog "why target verification can
 * be parallel" (all drafted positions are scored in one pass), TAPS §4.1 (the selected
 * subtree is verified with tree attention).
 *   out[b,h,i,:] = sum_j softmax_j(scale * q[b,h,i,:] . k[b,h/G,j,:]) v[b,h/G,j,:]
 *   with j over the prefix rows [0, P) and the tree rows {P + t : t in pi(i)},
 *   G = Hq / Hkv.
 *   q, out        [B][Hq][N][D]             dtype
 *   k_cache,
 *   v_cache       [B][Hkv][kv_stride_tokens][D] dtype; rows 0..P-1 = committed prefix,
 *                 row P + t = tree node t's key/value (already written by the caller;
 *                 keys are post-RoPE).  kv_stride_tokens >= P + N.
 *   parent        [B][N] int32
 *   scale         softmax scale (> 0); pass 0 for 1/sqrt(D).
 * Padding rows of a ragged batch: their rows of out are not written (the active rows'
 * results do not depend on the padding's q, k or v).
 * Precision: fp32 in/out with fp32 math, or bf16 in/out with fp32 softmax and fp32
 * accumulation.  Limits: 1 <= N <= 1024, 32 <= D <= 256 with D % 32 == 0, Hq % Hkv == 0.
 * bf16 with D in {64, 128}, G <= 16 and G * N >= 64 runs on the tensor cores; every
 * other case (fp32, other D, small trees) runs on the CUDA-core kernel.
 * Alignment: q, k_cache, v_cache, out 16-byte aligned.
 * Workspace (optional): tv_tree_attention_workspace_size(...) bytes, 16-byte aligned,
 * owned by the caller, device memory, no initial contents required.  It is nonzero only
 * where the plan is the persistent schedule (variant 4 of tv_set_attention_variant),
 * whose CTAs park partial rows of the units they share there; with a NULL or smaller
 * workspace that call runs the paired 64-key kernel (variant 3) unsplit instead, with
 * the same results up to fp32 summation order.  Split-KV partials of the other variants are merged through the
 * thread-block cluster's distributed shared memory.  Calls that share a workspace must
 * be ordered (one stream, or events).
 * Errors: NULL pointers -> TV_ERR_NULL; dtype -> TV_ERR_DTYPE; sizes, B * Hkv or the
 * grid outside the launch limits -> TV_ERR_SHAPE; scale < 0, NaN or infinite ->
 * TV_ERR_VALUE; misaligned pointers (workspace included) -> TV_ERR_ALIGN; a failed
 * launch -> TV_ERR_CUDA.  Tree structure problems
 * found on the device (node 0 not a root, or a parent index not below its node) and a
 * bounded wait that ran out are written to *dev_status.
 */
TV_API size_t tv_tree_attention_workspace_size(int B, int Hq, int Hkv, int D, int P, int N,
                                        tv_dtype dtype);
/* tv_tree_attention_plan - the kernel and KV split count that tv_tree_attention would use
 * for these sizes on the current device with the current settings
 * (tv_set_attention_variant, tv_set_attention_splits, tv_set_sm_partition):
 *   *kernel  0 CUDA-core kernel (fp32, or shapes the tensor-core kernels do not take),
 *            1 tensor-core kernel with one 128-row tile per CTA, 2 paired row tiles,
 *            3 paired row tiles with 64-key KV tiles and double-buffered S,
 *            4 variant 3 on a persistent grid (given the queried workspace),
 *            5 variant 3 on SM pairs
 *   *splits  KV ranges per tile group, merged in one thread-block cluster (1 for 4)
 * Automatic choice: the variant and split count that minimise a wave model of the run
 * time (waves of resident clusters x (KV tiles per CTA + fixed per-CTA and merge costs))
 * fitted to GB300 measurements.  Queries the device's cluster occupancy
 * (needs a current CUDA device); launches nothing.
 * Errors: NULL outputs -> TV_ERR_NULL; bad dtype -> TV_ERR_DTYPE; sizes -> TV_ERR_SHAPE.
 */
TV_API tv_status tv_tree_attention_plan(int B, int Hq, int Hkv, int D, int P, int N, tv_dtype dtype,
                                        int* kernel, int* splits);
TV_API tv_status tv_tree_attention(const void* q, const void* k_cache, const void* v_cache, void* out,
                            const int32_t* parent, int B, int Hq, int Hkv, int D, int P, int N,
                            int kv_stride_tokens, float scale, tv_dtype dtype, void* workspace,
                            size_t ws_bytes, int32_t* dev_status, tv_stream_t stream);

/* ------------------------------------------------------------------------------------
 * tv_verify_greedy - greedy acceptance of a draft tree.
 * Blog: "greedy decoding, intuitive version" and "accept a prefix and start the next
 * round": drafts are kept while they equal the target's choice; the first disagreement
 * is replaced by the target's token.
 * One streaming pass over the target logits computes, per row u: the argmax (lowest
 * index among equal raw values) and log-sum-exp of x/T with T = 1.  Then per sequence:
 * cur = root; while some child c of cur has tokens[c] == argmax[cur]: accept c, cur = c.
 *   logits        [B][N][V] dtype
 *   tokens        [B][N] int32 draft token of every node (tokens[b][0] unused)
 *   accepted_nodes[B][N] int32 out: accepted node ids in walk order, -1 padded
 *   accept_len    [B] int32 out: number of accepted drafts L (root excluded)
 *   bonus_token   [B] int32 out: argmax of the row where the walk stopped
 *   p_draft       [B][N] float out (optional): softmax(x[parent(c)])[tokens[c]], NaN at c=0
 *   row_lse       [B][N] float out (optional): log-sum-exp of each row
 *   row_argmax    [B][N] int32 out (optional): argmax of each row
 * Padding rows of a ragged batch: p_draft and row_lse NaN, row_argmax -1, never walked
 * (their logits are still read by the streaming pass).
 * Limits: 1 <= N <= 1024, 1 <= V < 2^31 / N, B * N <= 131072.
 * Workspace: tv_verify_workspace_size().
 */
TV_API size_t tv_verify_workspace_size(int B, int N, int V, tv_dtype dtype, int sampling);
TV_API tv_status tv_verify_greedy(const void* logits, const int32_t* parent, const int32_t* tokens, int B,
                           int N, int V, tv_dtype dtype, int32_t* accepted_nodes,
                           int32_t* accept_len, int32_t* bonus_token, float* p_draft,
                           float* row_lse, int32_t* row_argmax, void* workspace, size_t ws_bytes,
                           int32_t* dev_status, tv_stream_t stream);

/* ------------------------------------------------------------------------------------
 * tv_verify_greedy_static - tv_verify_greedy for callers that cannot allocate.
 * No counterpart in the paper: this is a packaging variant of tv_verify_greedy.  Some
 * callers cannot provide a workspace at call time - a plugin whose host framework owns
 * and plans all device memory, code running while a CUDA graph is being captured by a
 * component that forbids allocations, or runtimes that disallow allocation after
 * start-up.  This entry point takes the same inputs and outputs as tv_verify_greedy but
 * keeps its scratch in a fixed 4 MiB array inside the library's device image (every
 * GPU that loads the library holds it until exit).  It allocates nothing.
 *   - The first call on a device looks up that array's device address and zero-fills it
 *     synchronously; make that first call (per device) before any stream capture.
 *   - Each call clears the completion counters on `stream` before the vocab pass.
 *   - All calls share the array: calls that overlap on the GPU (other streams, other
 *     host threads) race and give undefined results.
 *   - Returns TV_ERR_WORKSPACE when the problem needs more scratch than the array holds:
 *     exactly when tv_verify_workspace_size(B, N, V, dtype, 0) exceeds 4194304 bytes.
 *     That size is about 72 bytes per logits row once B*N reaches 4096 rows (three
 *     16-byte partial slots plus six 4-byte per-row values), so B*N up to about 58,000
 *     rows fits; other errors as tv_verify_greedy.
 */
TV_API tv_status tv_verify_greedy_static(const void* logits, const int32_t* parent, const int32_t* tokens,
                                         int B, int N, int V, tv_dtype dtype, int32_t* accepted_nodes,
                                         int32_t* accept_len, int32_t* bonus_token, float* p_draft,
                                         float* row_lse, int32_t* row_argmax, int32_t* dev_status,
                                         tv_stream_t stream);

/* ------------------------------------------------------------------------------------
 * tv_vocab_stats - the fused vocabulary pass on its own, without an acceptance walk.
 * Blog "greedy decoding" and "acceptance probability for sampling": verification needs,
 * per node row u, the target's choice and the target (and draft) probability of each
 * drafted token.  One streaming read of the logits (and of the draft logits, when given)
 * computes, per row u of x/T: the argmax (lowest index among equal raw values) and the
 * natural-log log-sum-exp; per node c >= 1 the drafted token's probability in its
 * parent's row.  It is the pass that tv_verify_greedy and tv_verify_sample run before
 * their walks, exposed for callers that only want the statistics (acceptance rates,
 * their own walk) and to time the pass alone.
 *   logits        [B][N][V] dtype; draft_logits [B][N][V] dtype or NULL
 *   parent, tokens [B][N] int32 (tree layout above; tokens[b][0] unused)
 *   temperature   > 0; divides both logits arrays (argmax compares raw values)
 *   row_lse       [B][N] float out (optional): log-sum-exp of x/T per row
 *   row_argmax    [B][N] int32 out (optional): argmax per row
 *   p_draft       [B][N] float out (optional): softmax(x[parent(c)]/T)[tokens[c]], NaN at c=0
 *   draft_row_lse [B][N] float out (optional, needs draft_logits): lse of the draft rows
 *   q_draft       [B][N] float out (optional, needs draft_logits): the same gather in the
 *                 draft rows
 * Padding rows of a ragged batch: NaN lse and probabilities, argmax -1.
 * Limits as tv_verify_greedy.  Workspace: tv_verify_workspace_size(B, N, V, dtype,
 * draft_logits != NULL), zero-filled once; the call leaves it ready for the next one.
 * Errors: draft outputs without draft_logits -> TV_ERR_NULL; temperature <= 0 or not
 * finite -> TV_ERR_VALUE; others as tv_verify_greedy.
 */
TV_API tv_status tv_vocab_stats(const void* logits, const void* draft_logits, const int32_t* parent,
                                const int32_t* tokens, int B, int N, int V, float temperature, tv_dtype dtype,
                                float* row_lse, int32_t* row_argmax, float* p_draft, float* draft_row_lse,
                                float* q_draft, void* workspace, size_t ws_bytes, int32_t* dev_status,
                                tv_stream_t stream);

/* ------------------------------------------------------------------------------------
 * tv_verify_sample - stochastic acceptance down the draft tree.
 * Blog "acceptance probability for sampling": draft token t at node u is kept with
 * probability min(1, p_u(t)/q_u(t)); "how to correct after a rejection": the
 * replacement is drawn from (p-q)+ / sum (p-q)+.
 * p_u = softmax(target[u]/T), q_u = softmax(draft[u]/T).  At node u the children are
 * tried in ascending index order with uniforms U(seed, round, b, u, k, 0), k = 1..m;
 * after rejecting t_k: p <- (p-q)+ normalised (unchanged if the residual is 0) and
 * q <- q without t_k, renormalised.  When all children are rejected or u is a leaf, the
 * output token is the smallest v with U(seed, round, b, u, 0, 1) * sum(p) < p(0..v).
 * U is Philox4x32-10 (Salmon et al., SC'11) with key = seed and counter =
 * (round mod 2^32, b, u, 2k + kind), U = (x0 >> 8) * 2^-24.
 *   target_logits, draft_logits [B][N][V] dtype
 *   accepted_nodes [B][N], accept_len [B], out_token [B] int32 out
 *   p_draft, q_draft [B][N] float out (optional): p_{parent(c)}(t_c), q_{parent(c)}(t_c)
 * Padding rows of a ragged batch: p_draft and q_draft NaN, never tried.
 * Limits as tv_verify_greedy; temperature > 0.  Workspace:
 * tv_verify_workspace_size(B, N, V, dtype, 1).
 */
TV_API tv_status tv_verify_sample(const void* target_logits, const void* draft_logits,
                           const int32_t* parent, const int32_t* tokens, int B, int N, int V,
                           float temperature, uint64_t seed, uint64_t round, tv_dtype dtype,
                           int32_t* accepted_nodes, int32_t* accept_len, int32_t* out_token,
                           float* p_draft, float* q_draft, void* workspace, size_t ws_bytes,
                           int32_t* dev_status, tv_stream_t stream);

/* ------------------------------------------------------------------------------------
 * tv_commit_accepted_kv - keep the accepted root path's keys and values.
 * Blog, "KV cache handling": after verification only the accepted tokens' cache entries
 * stay in the target cache.  The tree's rows sit at P + t (root at P); for each sequence
 * b with L = accept_len[b] accepted nodes a_1..a_L (accepted_nodes[b][0..L-1], as
 * written by tv_verify_greedy / tv_verify_sample), row P + a_k of every KV head of both
 * caches is copied to row P + k, in place, so rows [0, P + L] become the cache of the
 * plain sequence prefix, root, a_1..a_L.  Other rows are left as they are.
 *   k_cache, v_cache [B][Hkv][kv_stride_tokens][D] (in/out), kv_stride_tokens >= P + N
 *   accepted_nodes [B][N] int32, accept_len [B] int32
 * Device checks: a_1 > 0, increasing, < N, and 0 <= L < N (TV_DEV_BAD_TREE otherwise;
 * that sequence's cache is then partly or not updated).  Host errors: NULL pointers,
 * sizes, D * element size not a multiple of 16 bytes or misaligned caches.
 * No workspace.
 */
TV_API tv_status tv_commit_accepted_kv(void* k_cache, void* v_cache, const int32_t* accepted_nodes,
                                const int32_t* accept_len, int B, int Hkv, int D, int P, int N,
                                int kv_stride_tokens, tv_dtype dtype, int32_t* dev_status,
                                tv_stream_t stream);

/* ------------------------------------------------------------------------------------
 * One single-drafter tree-expansion step (TreeGraft §3.1): the drafter ranks its
 * candidate pool by the cumulative path score s(v) and expands the frontier
 * F = Top_W(pool, s); each frontier node's next-token distribution contributes its
 * top-m tokens as children, with edge score p = the drafter's probability of the token
 * and path score s(child) = s(parent) * p.
 *
 * tv_frontier_topw: for each sequence b, the positions (into scores[b][0..count[b]-1])
 * of the W highest scores, highest first; ties go to the lower position.
 *   scores [B][C] float, count [B] int32 (<= C), out_idx [B][W] int32 (-1 past count).
 *   Limits: 1 <= C <= 4096, 1 <= W <= C.  count outside [0, C] -> TV_DEV_BAD_TREE.
 *
 * tv_expand_children: for each of R drafter rows (the next-token logits after a
 * frontier node), the top-m tokens (highest logit first, ties to the lower token id),
 * p = softmax(logits / temperature)[token] and s = fl32(parent_score[r] * p).
 *   draft_logits [R][V] (bf16 or fp32), parent_score [R] float,
 *   child_token [R][m] int32, child_p, child_score [R][m] float (token -1, p = s = 0
 *   where m > V).  Limits: 1 <= m <= 32.  temperature > 0.
 *   Workspace: tv_expand_workspace_size(R, V, m) bytes, zero-filled before first use.
 */
TV_API tv_status tv_frontier_topw(const float* scores, const int32_t* count, int B, int C, int W,
                           int32_t* out_idx, int32_t* dev_status, tv_stream_t stream);
TV_API size_t tv_expand_workspace_size(int R, int V, int m);
TV_API tv_status tv_expand_children(const void* draft_logits, const float* parent_score, int R, int V,
                             int m, float temperature, tv_dtype dtype, int32_t* child_token,
                             float* child_p, float* child_score, void* workspace, size_t ws_bytes,
                             int32_t* dev_status, tv_stream_t stream);

/* ------------------------------------------------------------------------------------
 * tv_select_subtree - budgeted prefix-closed subtree from a block-marginal pool.
 * TAPS §4.1: d positions x top-K tokens form the candidate tree (a node at depth k is a
 * rank path r_1..r_k with token pool_tokens[k-1][r_k]); TAPS §4.2: edge estimates are
 * propagated to a path-level reach probability and a prefix-closed subtree is kept under
 * a verification budget; TreeGraft §3.1: s(v) = product of the edge scores on the path.
 * Edge score := the child's marginal.  s is formed in fp32 left to right along the path
 * (correctly rounded multiplies).  The first budget-1 candidates in the order (s desc,
 * depth asc, rank path lexicographic asc) are kept; this set is prefix-closed and has
 * the largest sum of s among prefix-closed sets of its size.
 *   marg          [B][d][K] float, each position sorted by (prob desc, token asc), >= 0
 *   pool_tokens   [B][d][K] int32
 *   root_token    [B] int32 (device; may be NULL, the root's token is then -1)
 *   parent, tokens, depth [B][budget] int32 out, score [B][budget] float out: nodes in
 *                 selection order (parent < child), root = row 0 (score 1, depth 0);
 *                 rows past n_nodes hold -1 (score 0)
 *   n_nodes       [B] int32 out: 1 + number of selected candidates (may be NULL)
 * Limits: 1 <= d <= 16, 1 <= K <= 256, 1 <= budget <= 4096.
 * Workspace: tv_select_workspace_size(...) bytes (0 today: the kernel works in shared
 * memory; workspace may then be NULL).
 * Errors: NULL marg, pool_tokens or outputs -> TV_ERR_NULL; sizes -> TV_ERR_SHAPE;
 * ws_bytes below the query -> TV_ERR_WORKSPACE; a failed launch -> TV_ERR_CUDA.  A
 * marginal outside [0, 1] (NaN included) or a position not sorted by descending
 * marginal sets TV_DEV_BAD_TOKEN; pool tokens are copied to the output unchecked.
 */
TV_API size_t tv_select_workspace_size(int B, int d, int K, int budget);
TV_API tv_status tv_select_subtree(const float* marg, const int32_t* pool_tokens, int B, int d, int K,
                            int budget, const int32_t* root_token, int32_t* parent,
                            int32_t* tokens, int32_t* depth, float* score, int32_t* n_nodes,
                            void* workspace, size_t ws_bytes, int32_t* dev_status,
                            tv_stream_t stream);

/* ------------------------------------------------------------------------------------
 * tv_select_subtree_adaptive - tv_select_subtree cut to its cost-aware prefix.
 * TAPS §3.1 (limitation 2: verification latency grows with the selected node count)
 * and §3.2 (choose the compact prefix-closed subtree that maximises expected accepted
 * tokens per unit of verification cost instead of filling the budget).  Of the rows
 * tv_select_subtree(budget) would return, keeps the first n*, the smallest n in
 * [1, rows available] maximising
 *     (1 + sum_{i=1}^{n-1} score[i]) / (cost_base + cost_per_row * n)
 * where every score is first rounded to a multiple of 2^-40 and summed exactly, and
 * the ratio is an IEEE double division (so the choice does not depend on summation
 * order).  cost_base, cost_per_row: a line fitted to measured verification time
 * against tree rows (any unit, same for both).  Rows past n* hold -1 (score 0) and
 * n_nodes[b] = n*.  Other arguments, limits and workspace as tv_select_subtree, except
 * that n_nodes is required.
 * Handing the tree on: the rows past n_nodes[b] hold parent -1, the trailing padding
 * of a ragged batch, so parent and tokens go straight into tv_tree_prep,
 * tv_tree_attention, tv_verify_* and tv_vocab_stats with N = budget, every sequence
 * keeping its own node count.  The same holds for tv_select_subtree whenever the
 * candidate tree holds fewer than budget - 1 nodes.
 * Host errors: cost_base < 0, cost_per_row <= 0 or not finite -> TV_ERR_VALUE.
 */
TV_API tv_status tv_select_subtree_adaptive(const float* marg, const int32_t* pool_tokens, int B, int d,
                                     int K, int budget, float cost_base, float cost_per_row,
                                     const int32_t* root_token, int32_t* parent, int32_t* tokens,
                                     int32_t* depth, float* score, int32_t* n_nodes, void* workspace,
                                     size_t ws_bytes, int32_t* dev_status, tv_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* TREEVERIFY_H */
