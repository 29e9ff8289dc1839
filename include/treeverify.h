/*
 * libtreeverify -- the GPU hot path of tree-based speculative decoding on one
 * NVIDIA GB300 (sm_103a).
 *
 * One verify step of tree speculative decoding (OPT-Tree: Speculative Decoding
 * with Adaptive Draft Tree Structure, §2 Preliminaries; GOOSE: Anisotropic
 * Speculation Trees, §2C; Speculative Decoding concept page, "The protocol"):
 * a drafter proposes a tree of tokens, the target model scores every tree
 * node in one forward pass under a tree attention mask, and an acceptance rule
 * keeps the longest acceptable branch plus one token from the target.  This
 * library provides the data-parallel steps of that pass:
 *
 *   tv_tree_build     parent[] -> depth[], ancestor bitmasks (the tree mask)
 *   tv_attn_verify    GQA attention of every tree node over the KV prefix and
 *                     its own ancestors (one layer of the verify pass)
 *   tv_accept_greedy  longest branch matching the target's argmax sequence
 *   tv_accept_sample  stochastic acceptance min(1, p/q) with (p-q)+ residual
 *                     resampling, Philox4x64-10 random numbers
 *   tv_expand_gated   one layer of TALON's budget-driven, confidence-gated
 *                     tree expansion (root Top-K, anchor, alpha gate, budget)
 *   tv_expand_topn,   OPT-Tree's greedy expansion (one layer: the `width`
 *   tv_select_topn    best children of the frontier) and its subtree
 *                     selection (the n best nodes of the candidate tree)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *    its comment says otherwise.  The library keeps no state between calls
 *    and allocates no device memory; scratch comes from the caller's
 *    workspace argument, sized by the matching *_workspace_size() call.
 *  - Every call enqueues its kernels on `stream` and returns without waiting.
 *  - Errors the host can see (bad sizes, null pointers, unsupported shapes,
 *    a workspace that is too small) return a non-zero tv_status before
 *    anything is launched.  A failed kernel launch returns TV_ERR_CUDA.
 *  - Errors in device-resident data (a malformed parent[] array, a token
 *    outside [0, V), a kv_len that does not fit the cache) are written to the
 *    per-sequence `status[b]` array (0 = ok) and that sequence's outputs are
 *    set to -1 (indices) or 0 (values).  No kernel traps, asserts or
 *    spin-waits.
 *  - Trees: node 0 is the root (the token right after the cached prefix,
 *    always accepted), parent[b*N + 0] = -1 and 0 <= parent[b*N + i] < i for
 *    i > 0, i.e. the nodes are numbered in a topological order.  N <= 512.
 *  - Row v of a logits tensor is the distribution over the children of v.
 *  - bf16 tensors are passed as their 16-bit patterns (tv_bf16).
 *  - Workspaces marked "zero-filled" must be zero-filled before their first
 *    use (tv_workspace_clear) and are returned zero-filled by every call that
 *    completes.  Calls that share one workspace must not run concurrently.
 */
#ifndef TREEVERIFY_H_
#define TREEVERIFY_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t tv_bf16; /* IEEE bfloat16 bit pattern */

typedef enum {
  TV_OK = 0,
  TV_ERR_INVALID_ARG = 1,   /* bad size, null pointer, bad hyperparameter */
  TV_ERR_INVALID_TREE = 2,  /* parent[] is not a single-root topological tree */
  TV_ERR_UNSUPPORTED = 3,   /* shape outside the supported set (e.g. D not 64/128) */
  TV_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
  TV_ERR_TIMEOUT = 5,       /* reserved: a bounded device wait gave up */
  TV_ERR_INVALID_TOKEN = 6, /* a draft token outside [0, V) */
  TV_ERR_WORKSPACE = 7      /* workspace missing or smaller than required */
} tv_status;

/* Maximum tree size (nodes per sequence) handled by every entry point. */
#define TV_MAX_NODES 512

/* Human-readable name of a status code (static string, never NULL). */
const char* tv_status_string(tv_status s);

/* Library version as 10000*major + 100*minor + patch. */
int tv_version(void);

/* Zero-fill a workspace on `stream` (cudaMemsetAsync). */
tv_status tv_workspace_clear(void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * tv_tree_build -- encode draft trees as the tree attention mask.
 * (OPT-Tree §2 and §3: the target verifies all tree tokens in parallel using
 * a tree attention mask in which a node sees its ancestors and itself.)
 *
 *   parent    int32 [B, N]          parent of each node, see Conventions.
 *   depth     int32 [B, N]   out    depth[i] = edges from the root (root 0).
 *   anc_mask  uint64 [B, N, W] out  W = ceil(N / 64); bit (j % 64) of word
 *                                   j / 64 of node i is set iff j is i or an
 *                                   ancestor of i.
 *   status    int32 [B]      out    0, or TV_ERR_INVALID_TREE (then depth is
 *                                   -1 and anc_mask 0 for that sequence).
 * Requires 1 <= N <= TV_MAX_NODES, B >= 0 (B = 0 is a no-op).
 */
tv_status tv_tree_build(const int32_t* parent, int B, int N, int32_t* depth,
                        uint64_t* anc_mask, int32_t* status, cudaStream_t stream);

/*
 * tv_attn_verify -- one attention layer of the tree verify pass.
 * (OPT-Tree §2: all tree tokens are verified in one target pass under the tree
 * mask; GOOSE §2C: a single forward pass verifies the entire tree;
 * Speculative Decoding concept page, "Why it is a win": the pass reads the
 * KV cache once for all positions.)
 *
 * For sequence b, node i, query head h (kv head h / (Hq / Hkv)):
 *   out[b,i,h,:] = sum_j softmax_j(scale * q[b,i,h,:] . k[b,kvh,j,:]) v[b,kvh,j,:]
 * over the key slots j in {0 .. kv_len[b]-1} (the cached prefix) and
 * {kv_len[b] + a : a an ancestor of i or i itself} (the tree's own keys,
 * which the caller has written to the cache at slots kv_len[b] .. kv_len[b]+N-1).
 *
 *   q         bf16 [B, N, Hq, D]     queries (already rotary-embedded; node i
 *                                    sits at position kv_len[b] + depth[i]).
 *   k, v      bf16 [B, Hkv, Lcap, D] KV cache.  Slots >= kv_len[b] + N are
 *                                    never read into a result (their values
 *                                    may be anything, including NaN).
 *   kv_len    int32 [B]              prefix length of each sequence.
 *   anc_mask  uint64 [B, N, W]       from tv_tree_build.
 *   scale     softmax scale; 0 selects 1/sqrt(D).
 *   out       bf16 [B, N, Hq, D] out
 *   lse       float [B, N, Hq]   out natural-log normaliser log(sum_j exp(s_j));
 *                                    may be NULL.
 *   status    int32 [B] out          0, or TV_ERR_INVALID_ARG when kv_len[b] < 0
 *                                    or kv_len[b] + N > Lcap (outputs zeroed);
 *                                    may be NULL.
 *   workspace scratch of tv_attn_workspace_size() bytes, 256-byte aligned,
 *             any contents (not zero-filled; left holding the split-KV
 *             partials).  The size is 0 when the plan keeps each row tile's
 *             key range in one CTA; workspace may then be NULL.  Otherwise
 *             the key range of every 128-row tile is split over several CTAs
 *             and the call launches a second (merge) kernel; a workspace that
 *             is NULL, misaligned or smaller returns TV_ERR_WORKSPACE.  The
 *             partial rows are held as bf16 (the fp32 exponent range, so any
 *             finite bf16 value of v survives the split), with fp32 row
 *             maxima and sums.
 * Supported: D in {64, 128}; Hq % Hkv == 0; 1 <= N <= TV_MAX_NODES; Lcap >= N.
 */
size_t tv_attn_workspace_size(int B, int N, int Hq, int Hkv, int D, int Lcap);
/*
 * tv_attn_plan -- the launch plan tv_attn_verify takes for a shape (the pages
 * describe no kernels; this reports this library's own choice, for sizing and
 * testing).  Host only, launches nothing; the choice depends on the shape and
 * the current device's SM count (152 when no device can be queried).
 *   info  int32 [4] host out: query rows per CTA (128 or 256), node tiles per
 *         (sequence, kv head), splits of the key range, CTAs of the attention
 *         kernel.  With more than one split the merge kernel follows.
 * The environment variable TV_ATTN_PLAN="rows,splits" (rows 128 or 256,
 * splits from 1 to min(64, ceil(Lcap / 128))) overrides the choice for every
 * later call of tv_attn_plan, tv_attn_workspace_size and tv_attn_verify (for
 * tests and tuning; it is read on every call, so it must not change between
 * sizing a workspace and the call that uses it).  Other values are ignored.
 * Returns TV_ERR_INVALID_ARG for an unsupported shape, B = 0 or a NULL info.
 */
tv_status tv_attn_plan(int B, int N, int Hq, int Hkv, int D, int Lcap, int32_t* info);
tv_status tv_attn_verify(const tv_bf16* q, const tv_bf16* k, const tv_bf16* v,
                         const int32_t* kv_len, const uint64_t* anc_mask, int B, int N,
                         int Hq, int Hkv, int D, int Lcap, float scale, tv_bf16* out,
                         float* lse, int32_t* status, void* workspace, size_t ws_bytes,
                         cudaStream_t stream);

/*
 * tv_commit_path -- commit the accepted branch to the KV cache.
 * (Speculative Decoding concept page, "The protocol" step 4: the accepted
 * tokens and the correction become part of the prefix; OPT-Tree §2: the
 * accepted tokens form one root-to-node branch of the draft tree.)
 *
 * For sequence b with the accepted branch path[b, 0..a] (a = accept_len[b],
 * path[b, 0] = 0, as tv_accept_greedy and tv_accept_sample return it) and
 * every kv head h:
 *   k[b, h, kv_len[b] + d, :] <- k[b, h, kv_len[b] + path[b, d], :]   (d = 1..a)
 * and the same for v, after which the prefix holds a + 1 more tokens (node 0
 * and the accepted draft tokens; the correction or bonus token is the next
 * step's node 0):  new_kv_len[b] = kv_len[b] + a + 1.  Slots past
 * kv_len[b] + a keep whatever they held.
 *   k, v        bf16 [B, Hkv, Lcap, D] in/out, 16-byte aligned; D a multiple of 8.
 *   kv_len      int32 [B]   prefix length before the step.
 *   path        int32 [B, N], accept_len int32 [B]: the acceptance result.
 *   new_kv_len  int32 [B] out; must not be kv_len itself.
 *   status      int32 [B] out: 0, or TV_ERR_INVALID_ARG when accept_len[b] is
 *               outside [0, N - 1] (an acceptance that failed reports -1),
 *               the branch does not start at 0 or is not strictly increasing
 *               below N, or kv_len[b] + path[b, a] >= Lcap; that sequence's
 *               cache is left as it was and new_kv_len[b] = kv_len[b].
 * Device pointers owned by the caller; enqueued on `stream`; no workspace.
 */
tv_status tv_commit_path(tv_bf16* k, tv_bf16* v, const int32_t* kv_len, const int32_t* path,
                         const int32_t* accept_len, int B, int N, int Hkv, int D, int Lcap,
                         int32_t* new_kv_len, int32_t* status, cudaStream_t stream);

/*
 * tv_expected_accept -- expected acceptance length of a draft tree.
 * (OPT-Tree §3: a node's score is the product of the draft probabilities
 * along its path from the root, and the expected acceptance length is
 * approximated by the sum of the scores of the tree's nodes; the draft
 * trees of OPT-Tree, GOOSE and TALON can be compared by it.)
 *
 *   parent    int32 [B, N]  the tree (topological order, parent[0] = -1).
 *   prob      float [B, N]  draft probability of node i given its parent,
 *                           in [0, 1]; prob[b, 0] is not read.
 *   score     float [B, N] out, may be NULL: prod of prob over node i's path
 *                           (node 0 scores 1).
 *   expected  float [B] out: sum of score over nodes 1 .. N-1.
 *   status    int32 [B] out: 0, TV_ERR_INVALID_TREE, or TV_ERR_INVALID_ARG for
 *             a probability outside [0, 1] (outputs then 0).
 * fp32 products (at most ceil(log2 N) rounds deep per factor); the sum over
 * the draft nodes is reduced in fp32 per warp and fp64 across warps.
 */
tv_status tv_expected_accept(const int32_t* parent, const float* prob, int B, int N, float* score,
                             float* expected, int32_t* status, cudaStream_t stream);

/*
 * tv_build_spine_tree -- GOOSE anisotropic spine tree (host code, no GPU).
 * (GOOSE §2A: a deep chain of context-matched tokens, the spine, with wide
 * branches of transition tokens forking off every spine node, wider near the
 * root; §2B Proposition 2: branch allocation falling linearly with depth.)
 *
 *   spine_tokens   int32 [S]      host: the context-matched chain, in order.
 *   branch_tokens  int32 [Sb, K]  host: row j = candidates for a branch off
 *                                 spine node j (node 0 = the root), best
 *                                 first, -1 ends a row.
 *   root_token     token of node 0 (the last accepted token).
 *   budget         nodes in the tree, counting the root (>= 1).
 *   spine_ratio    in [0, 1]: the spine takes min(S, round(ratio (budget-1)))
 *                  nodes; the rest go to branch points j = 0 .. m-1
 *                  (m = min(spine + 1, Sb)) with widths proportional to m - j
 *                  (integer parts, then one each from the root), each capped
 *                  by its usable candidates (the spine's own token and
 *                  repeats skipped; a shortfall passes on to deeper points).
 *   parent, tokens int32 [budget] host out: the tree, breadth-first, the spine
 *                  child first at every depth; n_nodes host out: its size.
 * Returns TV_ERR_INVALID_ARG for negative sizes, budget < 1, a ratio outside
 * [0, 1] or a NULL pointer that is needed.
 */
tv_status tv_build_spine_tree(const int32_t* spine_tokens, int S, const int32_t* branch_tokens,
                              int Sb, int K, int root_token, int budget, float spine_ratio,
                              int32_t* parent, int32_t* tokens, int32_t* n_nodes);

/*
 * tv_spine_ratio_update -- GOOSE §2C: the spine ratio follows an exponential
 * moving average of the observed acceptance rate of the spine tokens:
 * returns clamp((1 - beta) ratio + beta observed, 0, 1).  Host code.
 */
float tv_spine_ratio_update(float ratio, float observed_accept_rate, float beta);

/*
 * tv_attn_verify_tree -- tv_tree_build and tv_attn_verify in one call (OPT-Tree
 * §2: the tree attention mask is derived from the draft tree; the same single
 * target pass verifies every node).  For trees of up to 64 nodes it is one
 * launch: every attention CTA builds the ancestor masks of its sequence in
 * shared memory from parent[], and the first CTA of each sequence also writes
 * depth, anc_mask and tree_status exactly as tv_tree_build would (an invalid
 * tree: depth -1, empty masks, TV_ERR_INVALID_TREE; the attention then runs
 * on those empty masks, as the two calls would).  Larger trees take the two
 * launches.  A model with several attention layers calls this for its first
 * layer of a step and tv_attn_verify with the returned masks for the others.
 *   parent       int32 [B, N]        in   as for tv_tree_build.
 *   q, k, v, kv_len, B, N, Hq, Hkv, D, Lcap, scale, out, lse, status,
 *   workspace, ws_bytes              as for tv_attn_verify (same workspace size).
 *   depth        int32 [B, N]        out  as tv_tree_build's depth.
 *   anc_mask     uint64 [B, N, W]    out  as tv_tree_build's masks.
 *   tree_status  int32 [B]           out  as tv_tree_build's status.
 * Outputs are identical, bit for bit, to tv_tree_build followed by
 * tv_attn_verify.  Errors as for those calls.
 */
tv_status tv_attn_verify_tree(const int32_t* parent, const tv_bf16* q, const tv_bf16* k,
                              const tv_bf16* v, const int32_t* kv_len, int B, int N, int Hq,
                              int Hkv, int D, int Lcap, float scale, tv_bf16* out, float* lse,
                              int32_t* status, int32_t* depth, uint64_t* anc_mask,
                              int32_t* tree_status, void* workspace, size_t ws_bytes,
                              cudaStream_t stream);

/*
 * tv_accept_greedy -- greedy acceptance over a verified tree.
 * (OPT-Tree §2: under greedy sampling the longest branch matching the target
 * model's highest-probability sequence is accepted; GOOSE §2C: unified greedy
 * walk over the tree.)
 *
 *   logits     float [B, N, V]  target logits; row i scores i's children.
 *   tokens     int32 [B, N]     draft token of each node (node 0's is unused).
 *   parent     int32 [B, N]     tree; depth int32 [B, N] from tv_tree_build.
 *   argmax     int32 [B, N] out first index of the row maximum (ties -> lowest).
 *   accept_len int32 [B] out    accepted draft tokens = depth[end].
 *   end_node   int32 [B] out    deepest node whose whole root path matches
 *                               (tokens[c] == argmax[parent[c]] on every edge);
 *                               ties -> lowest node index.
 *   path       int32 [B, N] out path[d] = the depth-d node on root..end, -1 after.
 *   bonus      int32 [B] out    argmax[end]: the target's own next token.
 *   status     int32 [B] out    0, TV_ERR_INVALID_TREE (parent/depth
 *                               inconsistent) or TV_ERR_INVALID_TOKEN.
 *   workspace  zero-filled, >= tv_accept_greedy_workspace_size(B, N, V) bytes.
 * Logits must be finite.  V >= 1.
 */
size_t tv_accept_greedy_workspace_size(int B, int N, int V);
tv_status tv_accept_greedy(const float* logits, const int32_t* tokens, const int32_t* parent,
                           const int32_t* depth, int B, int N, int V, int32_t* argmax,
                           int32_t* accept_len, int32_t* end_node, int32_t* path,
                           int32_t* bonus, int32_t* status, void* workspace,
                           size_t ws_bytes, cudaStream_t stream);

/*
 * tv_debug_set_wait_limit -- test hook for failure detection (the pages have
 * no counterpart).  Every wait of a kernel in this library is bounded: when
 * its limit (about a second of SM clock) runs out, the kernel stops waiting,
 * reports TV_ERR_TIMEOUT in status[b] and leaves with no copy in flight.
 * This call sets, for the current device, the limit of one such wait -- the
 * wait of tv_accept_greedy's CTAs for their logit chunks -- so that a test
 * can make it run out without a fault or a hang:
 *   cycles >= 1                 limit in SM cycles;
 *   cycles == 0                 a single non-blocking test of the copies
 *                               (a call then reports TV_ERR_TIMEOUT, since
 *                               its copies have only just been issued);
 *   cycles == TV_WAIT_LIMIT_DEFAULT  restores the regular limit.
 * The second wait that keeps copies from outliving a CTA keeps the regular
 * limit.  Host call, synchronous with respect to the device's default
 * stream; it must not overlap a tv_accept_greedy call on the device.
 * Returns TV_ERR_INVALID_ARG for other negative values.
 */
#define TV_WAIT_LIMIT_DEFAULT (-1LL)
tv_status tv_debug_set_wait_limit(long long cycles);

/*
 * Bounds-checked build (the pages have no counterpart; a debugging aid).
 * libtreeverify_checked.so is this library compiled with TV_CHECKED defined:
 * the same entry points, in which every index a kernel computes from its
 * inputs or its launch geometry is checked before the access it guards.  A
 * failed check skips that access (no trap, no fault) and records its site in
 * a device word of its source unit; results are then unspecified, but every
 * access stays inside the caller's buffers.  The attention kernel also
 * records there the site of a bounded wait that gave up, so that a
 * TV_ERR_TIMEOUT can be traced to the barrier it waited on.
 *
 * tv_checked_build      1 in the checked build, 0 in the regular one.
 * tv_debug_check_take   synchronises the current device, then writes to
 *                       *site the first failed check recorded since the
 *                       previous call, as (unit << 16) | source line, or 0
 *                       (always 0 in the regular build), and clears the
 *                       record.  Units: 1 tree, 2 greedy, 3 sample,
 *                       4 expand, 5 attention, 6 commit, 7 expected,
 *                       8 top-n selection, 9 library.  Host call; it must not
 *                       overlap a launch of this library on the device.
 *                       TV_ERR_INVALID_ARG if site is NULL, TV_ERR_CUDA if
 *                       the device reports an error.
 * tv_debug_check_selftest  test of the mechanism itself: writes buf[i] = i for
 *                       i < n, each store guarded by the check
 *                       0 <= i < logical_n.  buf: device int32 [n], caller-
 *                       owned.  The regular build writes all n entries; the
 *                       checked build writes the first min(n, logical_n) and,
 *                       if n > logical_n, records a failed check (unit 9).
 *                       Every store lies inside buf either way.
 */
int tv_checked_build(void);
tv_status tv_debug_check_take(int32_t* site);
tv_status tv_debug_check_selftest(int32_t* buf, int n, int logical_n, cudaStream_t stream);

/*
 * tv_accept_greedy_noalloc -- tv_accept_greedy without a workspace.
 * The method description has no counterpart for this call: it exists for
 * callers that cannot allocate device memory where they run acceptance (a
 * serving loop whose memory plan is fixed at start-up, a plug-in that is
 * handed no allocator, a real-time path that must not allocate).
 *
 * Same arguments, outputs and status codes as tv_accept_greedy, minus the
 * workspace.  Scratch (one 64-bit key per node row, one counter per
 * sequence) lives in a fixed array of 528 KiB inside the library, present on
 * every GPU that loads it until the process exits.  Limits: B * N <= 65536
 * and B <= 4096; larger calls return TV_ERR_UNSUPPORTED without launching.
 * The call allocates nothing: it clears the part of the array it uses
 * (cudaMemsetAsync on `stream`) and launches the greedy kernel.
 * Every call on a device shares that array, so calls whose kernels may
 * overlap on the GPU (different streams, no ordering between them) race and
 * must not be issued.  The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture.
 */
tv_status tv_accept_greedy_noalloc(const float* logits, const int32_t* tokens,
                                   const int32_t* parent, const int32_t* depth, int B, int N,
                                   int V, int32_t* argmax, int32_t* accept_len, int32_t* end_node,
                                   int32_t* path, int32_t* bonus, int32_t* status,
                                   cudaStream_t stream);

/*
 * tv_accept_sample -- stochastic (lossless) acceptance over a verified tree.
 * (Speculative Decoding concept page, "The protocol" step 3: accept a draft
 * token x with probability min(1, p(x)/q(x)); on rejection resample from the
 * normalised (p - q)+; the output is distributed exactly as the target.)
 *
 * p = softmax(p_logits / T), q = softmax(q_logits / T) per node row.  Walk
 * from the root with r = p_root: test the children of the current node in
 * ascending index; child c with token x is accepted iff u < r(x) / q(x)
 * (always when q(x) = 0); accepting descends to c with r = p_c; a rejection
 * replaces r by (r - q)+ / sum((r - q)+) (kept when that sum is not positive).
 * When all children are rejected out_token is drawn from r; at a leaf it is
 * drawn from p_leaf (the bonus token).  Draws are inverse-CDF in ascending
 * token order.
 *
 * Random numbers: Philox4x64-10 (Salmon et al., "Parallel Random Numbers:
 * As Easy as 1, 2, 3", SC'11), key (seed, 0), counter (offset, b, node,
 * purpose << 32 | ordinal) with purpose 0 = accept test of the ordinal-th
 * child, 1 = the final draw; u = (first output word >> 11) * 2^-53.
 * (seed, offset) fully determine the result: advance offset between steps.
 *
 *   p_logits, q_logits float [B, N, V]; tokens, parent, depth int32 [B, N].
 *   temperature > 0.
 *   accept_len, end_node, out_token int32 [B] out; path int32 [B, N] out;
 *   status int32 [B] out (as tv_accept_greedy).
 *   workspace unused: tv_accept_sample_workspace_size() returns 0 and
 *             workspace may be NULL (each sequence's walk keeps its state in
 *             the shared memory of one thread-block cluster).
 * Supported: V <= 409,600 (a cluster's shared memory holds the visited row
 * pair); larger vocabularies return TV_ERR_UNSUPPORTED.
 */
size_t tv_accept_sample_workspace_size(int B, int N, int V);
tv_status tv_accept_sample(const float* p_logits, const float* q_logits,
                           const int32_t* tokens, const int32_t* parent,
                           const int32_t* depth, int B, int N, int V, float temperature,
                           uint64_t seed, uint64_t offset, int32_t* accept_len,
                           int32_t* end_node, int32_t* path, int32_t* out_token,
                           int32_t* status, void* workspace, size_t ws_bytes,
                           cudaStream_t stream);

/*
 * tv_expand_gated -- one layer of TALON tree expansion.
 * (TALON: confidence-aware speculative decoding with adaptive token trees,
 * §5.1 token budget B = maximum nodes in the tree; §5.2.2 layer 1 is the
 * Top-K of the root's draft distribution; §5.2.1 deeper layers: candidate
 * pool = all children of the frontier, path score s(c) = product of draft
 * probabilities, anchor = max s, keep s >= alpha * s_anchor, and when more
 * survive than the remaining budget keep the highest-scoring ones.)
 *
 *   draft_logits      float [F, V]  draft logits of the F frontier nodes.
 *   frontier_node     int32 [F]     their node ids (ascending).
 *   frontier_logscore float [F]     their log path scores (root: 0).
 *   layer             1 (Top-K of the single root row, F must be 1) or >= 2.
 *   topk, alpha       K (layer 1) and the gate 0 < alpha <= 1 (layers >= 2).
 *   budget            maximum nodes in the tree, counting the root.
 *   tree_parent, tree_token int32 [budget], tree_logscore float [budget]:
 *                     the kept candidates are appended at ids n_nodes.. in
 *                     (parent asc, score desc, token asc) order; ties in the
 *                     budget cut go to (parent asc, token asc).
 *   n_nodes           int32 [1], device, in/out: nodes in the tree.
 *   workspace         >= tv_expand_workspace_size(F, V) bytes, zero-filled before
 *                     its first use; every call returns its control words (per-row
 *                     arrival counters, candidate count, anchor, the floor's
 *                     histogram) to zero, so the same workspace serves the next
 *                     call as it is.
 * Three launches: per-row statistics (the last CTA of a row forms the row's
 * normaliser and raises the anchor), the gate filter, the budget select.  The
 * root layer's Top-K also gets a floor under its cut from the chunk maxima:
 * found in the statistics pass when the row has at least `topk` chunks of
 * 2048 logits, else by a fourth launch before the filter.
 * Scores are compared in fp64 (log domain) from fp32 logits.
 */
size_t tv_expand_workspace_size(int F, int V);
tv_status tv_expand_gated(const float* draft_logits, const int32_t* frontier_node,
                          const float* frontier_logscore, int F, int V, int layer, int topk,
                          float alpha, int budget, int32_t* tree_parent, int32_t* tree_token,
                          float* tree_logscore, int32_t* n_nodes, void* workspace,
                          size_t ws_bytes, cudaStream_t stream);

/*
 * tv_expand_topn -- one layer of OPT-Tree's greedy tree expansion.
 * (OPT-Tree §3: a node's score is the product of the draft probabilities
 * along its path; the frontier nodes are expanded and the layer keeps the
 * highest-scoring children, which are the next frontier.)
 *
 *   draft_logits      float [F, V]  draft logits of the F frontier nodes.
 *   frontier_node     int32 [F]     their node ids (ascending).
 *   frontier_logscore float [F]     their log path scores (root: 0).
 *   width             children kept by the layer, 1..2048: the best ones over
 *                     all F x V candidates (log score = the parent's + the
 *                     child's log-softmax value), ties to the lower
 *                     (parent, token).  F <= 2048.
 *   capacity          length of the tree arrays; the layer keeps
 *                     min(width, F x V, capacity - n_nodes) children, a number
 *                     the host can know without reading the device.
 *   tree_parent, tree_token int32 [capacity], tree_logscore float [capacity]:
 *                     the kept children are appended at ids n_nodes.. in
 *                     (parent asc, score desc, token asc) order.
 *   n_nodes, workspace as for tv_expand_gated (the same workspace layout and
 *                     size, tv_expand_workspace_size(F, V), zero-filled before
 *                     its first use and returned zero-filled).
 * The same three launches as tv_expand_gated, without the gate.  The floor
 * under the layer's cut comes from the chunk maxima: in the statistics pass
 * when the frontier has at least `width` chunks of 2048 logits, else by a
 * fourth launch before the filter; a chunk that holds more than `width`
 * candidates raises it further, so that later chunks pass on only what can
 * still be kept.
 */
tv_status tv_expand_topn(const float* draft_logits, const int32_t* frontier_node,
                         const float* frontier_logscore, int F, int V, int width, int capacity,
                         int32_t* tree_parent, int32_t* tree_token, float* tree_logscore,
                         int32_t* n_nodes, void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * tv_select_topn -- OPT-Tree's subtree selection: the n best nodes.
 * (OPT-Tree §3: keep the n highest-scoring nodes of the candidate tree; as a
 * node never scores above its parent, they form a subtree containing the
 * root, the one of n nodes with the largest expected acceptance length.)
 *
 *   parent, token int32 [B, M], logscore float [B, M]: B candidate trees
 *                 (topological order, parent[0] = -1), M <= 16384.
 *   n_nodes       int32 [B]: nodes in use per tree, 1..M.
 *   n             nodes to keep (>= 1); ties go to the lower node id.
 *   out_parent, out_token, out_src int32 [B, n], out_logscore float [B, n]:
 *                 the kept nodes renumbered in their original order (still
 *                 topological); out_src = a node's id in the input.  Rows
 *                 k .. n-1, k = min(n, n_nodes[b]), are -1 (0 for scores).
 *   expected      float [B]: sum of exp(logscore) over the kept nodes other
 *                 than the root (OPT-Tree's expected acceptance length).
 *   status        int32 [B]: 0; TV_ERR_INVALID_TREE for a malformed parent
 *                 array or a kept node whose parent was not kept (scores that
 *                 rise along a path); TV_ERR_INVALID_ARG for a NaN score or
 *                 n_nodes outside 1..M.  The outputs of such a tree are -1 / 0.
 * One CTA per tree: a radix select of the score keys in shared memory, then
 * block scans over the ids.  Scores are compared as fp32 values (-0 = +0).
 */
tv_status tv_select_topn(const int32_t* parent, const int32_t* token, const float* logscore,
                         const int32_t* n_nodes, int B, int M, int n, int32_t* out_parent,
                         int32_t* out_token, float* out_logscore, int32_t* out_src,
                         float* expected, int32_t* status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TREEVERIFY_H_ */
