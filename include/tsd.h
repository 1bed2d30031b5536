/*
 * tsd.h -- C ABI of the tree-speculative-decoding verify path (libtsd.so).
 *
 * The library runs, on one GPU, the target model's verification of a draft
 * tree: safe ancestor tables with a virtual root, tree-masked attention over a
 * paged KV cache, greedy longest-accepted-path search, and the fast-reorder
 * commit of the accepted K/V.  An optional entry point builds best-first
 * budgeted draft trees from per-position marginals.
 *
 * Sources (page title, section):
 *   [EP-zh]   "EAGLE-Pangu: Accelerator-Safe Tree Speculative Decoding on
 *             Ascend NPUs", technical summary (gist.science/zh/paper/2603.08088),
 *             2.1 branchable KV cache, 2.2 accelerator-safe tree tensor
 *             semantics, 2.3 fused tree-masked teacher execution.
 *   [EP-pt]   the same paper's Portuguese technical summary, section 2.
 *   [BASTION] "Resumo Técnico: BASTION" (gist.science/pt/paper/2605.29727),
 *             Methodology 1 and 2.
 *   [Blog]    "Speculative Decoding Hierárquico: Medusa, EAGLE-2 e
 *             Multi-Token Prediction" (produtoramaxvision.com.br), sections
 *             on Medusa tree attention and on vLLM PagedAttention.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * - Every array argument is a DEVICE pointer to memory the caller owns and
 *   allocated.  The library allocates nothing, frees nothing and never
 *   synchronises: all work is enqueued on `stream` (a cudaStream_t; NULL is
 *   the legacy default stream) in launch order, and results are ready when
 *   the stream reaches that point.
 * - Kernels are launched with programmatic dependent launch: a kernel may
 *   start while the previous kernel on the stream is still running, if that
 *   kernel is one of this library's and releases its dependents early (every
 *   kernel here does, except the commits, which release only when they end).
 *   Each kernel waits for the previous one before it reads that kernel's
 *   results and before its first global write.  tsd_tree_attn_fwd under the
 *   uniform split reads its inputs (q, the caches, block table, lengths,
 *   records) before that wait, and the mask and err after it: a library
 *   kernel just before it must therefore not write those inputs, which holds
 *   for tsd_tree_build_ancestors (the usual predecessor).
 * - Return value: a host-detected status (TSD_OK or a negative TSD_ERR_*).
 *   On a non-zero return nothing was launched (TSD_ERR_CUDA: a launch failed;
 *   the CUDA error is left for the caller to query).
 * - Problems the host cannot see (device-resident lengths, block ids, paths)
 *   are reported on the device: per-sequence error bits in err[b], and a
 *   device status word `status` (OR of TSD_STATUS_* bits; the caller zeroes it
 *   when it wants a fresh reading).  Such sequences are skipped, never read or
 *   written out of bounds (fail closed).
 * - Node ids: callers give real ids 0..N_b-1; node 0 is the tree root (the
 *   last emitted token, whose K/V is the first tree slot) with parent -1.
 *   Tables built by the library use safe ids s = i + 1 with the virtual root at
 *   0, so every gather index lies in [0, N_max] ([EP-zh] 2.2).
 * - bf16 arrays are passed as uint16_t bit patterns.
 * - KV cache: paged, 16 token slots per block, layout
 *   [num_blocks][Hkv][16][D]; token slot t of sequence b lives in block
 *   block_table[b * max_blocks + t / 16], row t % 16.  Sequence b's committed
 *   prefix is slots [0, P_b); the draft tree's own K/V sit at slot P_b + i for
 *   real node i ([EP-zh] 2.1 committed vs speculative state; [Blog] paged
 *   blocks).
 * - Limits (TSD_ERR_LIMIT): 1 <= N_max <= 256, 0 <= D_max <= 32,
 *   D in {64, 128}, Hq % Hkv == 0, Hq / Hkv <= 16, B <= 65535.
 */
#ifndef TSD_H_
#define TSD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *tsd_stream_t; /* same handle as cudaStream_t */

/* host-detected status */
enum {
  TSD_OK = 0,
  TSD_ERR_ARG = -1,       /* null pointer, negative size, misaligned pointer */
  TSD_ERR_LIMIT = -2,     /* a size outside the limits listed above */
  TSD_ERR_WORKSPACE = -3, /* workspace missing or smaller than required */
  TSD_ERR_CUDA = -4       /* a kernel launch failed */
};

/* err[b] bits written by tsd_tree_build_ancestors ([EP-zh] 2.2 checks) */
#define TSD_TREE_RANGE 1   /* non-root parent outside [0, N_max) (incl. a second -1) */
#define TSD_TREE_CYCLE 2   /* walking up from a node does not reach the root */
#define TSD_TREE_TOO_DEEP 4 /* a node deeper than D_max */
#define TSD_TREE_CLOSURE 8 /* a valid node whose parent is a padding node */
#define TSD_TREE_ROOT 16   /* parent[0] != -1 */
#define TSD_TREE_COUNT 32  /* n_nodes[b] outside [1, N_max] */

/* device status word bits */
#define TSD_STATUS_BAD_PAGE 1 /* a block id outside [0, num_blocks): sequence skipped */
#define TSD_STATUS_BAD_LEN 2  /* P_b < 0 or P_b + N_b beyond max_slots / the table */
#define TSD_STATUS_BAD_PATH 4 /* accept_len / path inconsistent with the tree */
#define TSD_STATUS_TIMEOUT 8  /* a bounded wait inside a kernel ran out: outputs unspecified */

/* Library version string (static storage). */
const char *tsd_version(void);

/*
 * Process-wide options (host state, read at each launch; not thread-safe
 * against concurrent launches).  No page counterpart: they exist for tests
 * and measurement.
 *   TSD_OPT_WAIT_LIMIT_NS  limit of every bounded wait inside a kernel, in
 *                          ns (default 2e9).  When a wait runs out the kernel
 *                          sets TSD_STATUS_TIMEOUT, drains its in-flight copies
 *                          and MMAs (bounded), frees its tensor memory and
 *                          returns; 0 makes every wait that is not already
 *                          satisfied run out.
 *   TSD_OPT_TEST_STALL     1: the tcgen05 attention's MMA thread first waits
 *                          on a barrier nothing ever signals, so that wait
 *                          runs out after TSD_OPT_WAIT_LIMIT_NS and the
 *                          timeout path runs (tests only; default 0).
 * Returns TSD_ERR_ARG for an unknown key or value.
 */
#define TSD_OPT_WAIT_LIMIT_NS 0
#define TSD_OPT_TEST_STALL 1
#define TSD_OPT_COUNT 2
int tsd_set_option(int key, int64_t value);
int64_t tsd_get_option(int key);

/*
 * a1. Accelerator-safe tree tensors ([EP-zh] 2.2; [EP-pt] section 2,
 *     "Semântica de Tensores em Árvore Segura").
 *
 * Replaces the root's -1 sentinel by a virtual root row 0, builds the
 * ancestor index table, the per-node ancestor bitmask and the depth, and runs
 * the range / acyclicity / validity-closure checks before any fused kernel.
 *
 * parent   int32 [B][N_max]  real ids; parent[b][0] must be -1; entries of
 *                             padding nodes (i >= n_nodes[b]) are ignored.
 *                             Any order is allowed (no topological order).
 * n_nodes  int32 [B] or NULL (NULL: every sequence has N_max nodes).
 * anc      int32 [B][N_max+1][D_max+1]  out.  anc[b][s][d] = safe id of the
 *                             depth-d ancestor of safe node s (d <= depth),
 *                             0 beyond; row 0 (virtual root) and padding rows
 *                             are all 0.
 * depth    int32 [B][N_max]  out.  depth(root) = 0; padding rows 0.
 * mask     uint32 [B][N_max][W], W = ceil(N_max / 32)  out.  Bit j of row i is
 *                             set iff real node j is i or an ancestor of i.
 * err      int32 [B]  out.  OR of TSD_TREE_* bits; a sequence with err != 0
 *                             gets all-zero rows and is skipped by the other
 *                             entry points.
 * One thread block per sequence.
 */
int tsd_tree_build_ancestors(const int32_t *parent, const int32_t *n_nodes, int B, int N_max,
                             int D_max, int32_t *anc, int32_t *depth, uint32_t *mask, int32_t *err,
                             tsd_stream_t stream);

/*
 * a2. Tree-masked attention for all tree nodes in one pass ([EP-zh] 2.3:
 *     node k attends only to its ancestor path and itself, no cross-branch
 *     leakage; [Blog] Medusa tree attention mask).
 *
 * For every valid (b, node i, q head h):
 *   out = softmax(scale * q . K^T) V over the keys of kv head h / (Hq/Hkv):
 *   every prefix slot [0, P_b), plus tail slot P_b + j iff bit j of
 *   mask[b][i] is set.  fp32 accumulation, out rounded to bf16 (nearest
 *   even).  lse (optional) = natural log of the sum of exp(scale * q . k).
 * No positional rotation is applied (rotate q/k with position P_b + depth).
 *
 * q           bf16 [B][N_max][Hq][D]
 * k_cache,
 * v_cache     bf16 [num_blocks][Hkv][16][D]   (see conventions)
 * block_table int32 [B][max_blocks]
 * prefix_len  int32 [B]   P_b
 * n_nodes     int32 [B] or NULL
 * mask        uint32 [B][N_max][W]   from tsd_tree_build_ancestors
 * err         int32 [B] or NULL      sequences with err != 0 are skipped
 * max_slots   host upper bound on P_b + N_b over the batch, at most 262144
 *             (TSD_ERR_LIMIT beyond); it sizes the split-KV grid and the
 *             workspace.  A sequence exceeding it sets TSD_STATUS_BAD_LEN
 *             and is skipped.  For batches of up to 64 sequences the key
 *             ranges are split on the device from the actual lengths, so a
 *             loose bound costs workspace, not time.
 * out         bf16 [B][N_max][Hq][D]  out.  Skipped / padding rows are 0.
 * lse         float [B][N_max][Hq] or NULL  out.  Skipped rows -inf.
 * workspace   device scratch of ws_bytes >= tsd_tree_attn_workspace_bytes()
 *             (split-KV partials and the split plan; no initial contents
 *             required).  That size is 0, and workspace may be NULL, when
 *             every key range is one piece (below).
 * status      int32 device word (see TSD_STATUS_*), may be NULL.
 * Work split: the key range of each (sequence, kv head, block of 128 or 256
 * query rows) is cut into pieces sized to fill the GPU; a second kernel
 * merges the pieces of each row.  When every range is one piece the rows are
 * written directly: one launch, no workspace.  Batches of 2..64 sequences
 * whose blocks would walk long key ranges are split on the device from the
 * actual lengths (three launches: plan, split, merge).
 */
size_t tsd_tree_attn_workspace_bytes(int B, int N_max, int Hq, int Hkv, int D, int max_slots);
/* Kernels one tsd_tree_attn_fwd call launches for these sizes on the current
 * device (1: one piece per key range; 2: split + merge; 3 with the device-side
 * split plan); 0 for sizes it rejects.  Host only. */
int tsd_tree_attn_launches(int B, int N_max, int Hq, int Hkv, int D, int max_slots);
/* The launch shape tsd_tree_attn_fwd picks for these sizes on the current
 * device (host only; for measurement and tests).  info: int32 [8] out:
 * mode (1: uniform split, 2: device plan), two-blocks-per-SM kernel (0/1),
 * query rows per block (128 or 256), row blocks per kv head, pieces per key
 * range (mode 2: the uniform guess the plan refines), keys per piece, blocks
 * in the grid, and 1 when rows go straight to the output (one piece, no
 * merge kernel).  TSD_ERR_LIMIT / TSD_ERR_ARG as tsd_tree_attn_fwd. */
int tsd_tree_attn_plan(int B, int N_max, int Hq, int Hkv, int D, int max_slots, int32_t *info);
int tsd_tree_attn_fwd(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                      const int32_t *block_table, int max_blocks, int num_blocks,
                      const int32_t *prefix_len, const int32_t *n_nodes, const uint32_t *mask,
                      const int32_t *err, int B, int N_max, int Hq, int Hkv, int D, int max_slots,
                      float scale, uint16_t *out, float *lse, void *workspace, size_t ws_bytes,
                      int32_t *status, tsd_stream_t stream);

/*
 * a2 through a deferred commit (see tsd_kv_commit_remap): the same attention
 * over the committed sequence of length P_b = prefix_len[b] and the tree,
 * where
 *   - logical slot s in [remap_base[b], remap_base[b] + remap_len[b]) is read
 *     from physical slot remap_src[b * remap_stride + s - remap_base[b]];
 *   - the tree's node j is read from physical slot tail_base[b] + j;
 *   - every other slot is read where it is.
 * Keys are visited in logical order, so the result is bit for bit the one
 * tsd_tree_attn_fwd gives after the copy commit moved the same entries.
 * remap_src/remap_base/remap_len: all NULL (no record) or all given, with
 * 1 <= remap_stride <= 33 and each record inside [0, P_b) (else the sequence
 * is skipped with TSD_STATUS_BAD_LEN); tail_base NULL: the tree at P_b.
 * Recorded slots and the tree are fetched slot by slot, the rest of the key
 * range with the usual block loads.  Other arguments as tsd_tree_attn_fwd.
 */
int tsd_tree_attn_fwd_remap(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                            const int32_t *block_table, int max_blocks, int num_blocks,
                            const int32_t *prefix_len, const int32_t *n_nodes,
                            const uint32_t *mask, const int32_t *err, int B, int N_max, int Hq,
                            int Hkv, int D, int max_slots, float scale, const int32_t *remap_src,
                            int remap_stride, const int32_t *remap_base, const int32_t *remap_len,
                            const int32_t *tail_base, uint16_t *out, float *lse, void *workspace,
                            size_t ws_bytes, int32_t *status, tsd_stream_t stream);

/*
 * a3. Greedy verification ([Blog] Medusa: the target evaluates every branch
 *     in one parallel pass and the longest valid path is selected; [EP-zh]
 *     lay summary section 3).
 *
 * argmax[b][i] = first index of the maximum of logits[b][i][0..V) (exact fp32
 * compares, lowest index on ties, +0 == -0).  Acceptance: the root is
 * accepted; node i is accepted iff its parent is and tokens[b][i] ==
 * argmax[b][parent(i)].  leaf = deepest accepted node (lowest id on ties);
 * accept_len = depth(leaf); path[b][k] = anc[b][leaf+1][k] for k <= accept_len,
 * 0 beyond (the kernel walks the leaf's parents, which gives the same row of
 * a table built by tsd_tree_build_ancestors from the same parent array);
 * bonus = argmax[b][leaf].
 *
 * logits  float [B][N_max][V]; tokens, parent int32 [B][N_max];
 * anc, depth, mask, err  from tsd_tree_build_ancestors; n_nodes int32 [B] or NULL.
 * argmax  int32 [B][N_max] out (-1 for padding rows and skipped sequences);
 * accept_len, leaf, bonus int32 [B] out; path int32 [B][D_max+1] out.
 * A sequence with err != 0: accept_len 0, leaf -1, bonus -1, path 0.
 * workspace  >= tsd_tree_verify_workspace_bytes() bytes (a ticket per
 *            sequence and a 64-bit argmax key per row), ZERO-FILLED before
 *            its first use; every call leaves it zero-filled again.  Calls
 *            sharing one workspace must not overlap on the GPU.
 * One fused launch: each sequence's rows are streamed in equal ranges, one
 * per block, and the block that retires a sequence's last range runs its
 * acceptance search.
 */
size_t tsd_tree_verify_workspace_bytes(int B, int N_max, int V);
int tsd_tree_verify_greedy(const float *logits, const int32_t *tokens, const int32_t *parent,
                           const int32_t *anc, const int32_t *depth, const uint32_t *mask,
                           const int32_t *n_nodes, const int32_t *err, int B, int N_max, int V,
                           int D_max, int32_t *argmax, int32_t *accept_len, int32_t *leaf,
                           int32_t *path, int32_t *bonus, void *workspace, size_t ws_bytes,
                           tsd_stream_t stream);

/*
 * Allocation-free variant of tsd_tree_verify_greedy (the pages have no
 * counterpart; it exists for callers that cannot allocate device memory).
 *
 * Some callers cannot call cudaMalloc: a plugin inside another engine that
 * owns all device memory and offers no workspace, or a latency-critical path
 * where an allocation, which may synchronise the device, is not allowed.
 * This call takes the same arguments and produces the same results as
 * tsd_tree_verify_greedy, without a workspace: its scratch is a fixed array
 * of tsd_tree_verify_static_capacity() bytes (1 MiB) in device memory that
 * every GPU loading the library holds until the process exits.  Sizes whose
 * scratch (B tickets plus B * N_max 8-byte argmax keys) exceeds it return
 * TSD_ERR_LIMIT.  The call itself allocates nothing.
 * - The first call on a device looks up the array's device address (with
 *   that device current) and caches it with the id of the device's context;
 *   a call after a device reset looks it up again.  Make the first call on a
 *   device (and the first after a reset) before any stream capture.  Host
 *   threads may call concurrently: the look-up is serialised.
 * - Every call zeroes the tickets and keys it uses on `stream` before its
 *   kernel runs.
 * - Each GPU has its own instance of the array.  All calls on one device
 *   share it: calls that overlap on the same device (two streams) race.
 */
size_t tsd_tree_verify_static_capacity(void);
int tsd_tree_verify_greedy_static(const float *logits, const int32_t *tokens,
                                  const int32_t *parent, const int32_t *anc, const int32_t *depth,
                                  const uint32_t *mask, const int32_t *n_nodes, const int32_t *err,
                                  int B, int N_max, int V, int D_max, int32_t *argmax,
                                  int32_t *accept_len, int32_t *leaf, int32_t *path,
                                  int32_t *bonus, tsd_stream_t stream);

/*
 * Stochastic verification ([Blog], classic speculative decoding: modified
 * rejection sampling accepts a drafted token x ~ q with probability
 * min(1, p(x)/q(x)) and on rejection draws from the normalised residual
 * max(0, p - q), so the emitted token is distributed as the target p;
 * [Blog] Medusa: every branch of the tree scored in one pass).
 *
 * Tree reading: the children of node i are independent draws from q_i (row i
 * of q_draft), tried in increasing id order.  With p_i = softmax(logits[i])
 * and r = p_i, child c (token x) is accepted iff
 *   u_accept[b][c] * q_i(x) < r(x);
 * on rejection r <- max(0, r - q_i) / sum(max(0, r - q_i)) (r <- q_i when
 * that sum is 0) and the next child is tested.  A node whose children are
 * all rejected draws draw[b][i] from r by inverse CDF in token order: the
 * first token whose cumulative weight exceeds u_draw[b][i] times the total
 * (rounding leaving none: the last token of positive weight).  A walk that
 * ends at a leaf draws the leaf's token the same way from p_leaf.
 * Children whose token lies outside [0, V) are skipped.  The walk starts at
 * the root and follows next[] to the first node without an accepted child:
 * accept_len = its depth, leaf = it, bonus = its draw, path[b][k] = safe id
 * of the depth-k node of the walk, 0 beyond (the same layout as
 * tsd_tree_verify_greedy, so tsd_kv_commit_path takes the result as is).
 * Arithmetic is fp32 (max, sums, exponentials, residuals); each decision
 * matches the exact one unless its uniform lies within rounding of the
 * threshold.
 *
 * logits, q_draft  float [B][N_max][V]  target logits and draft
 *                  probabilities (rows need not be normalised; non-negative,
 *                  finite; logits finite or -inf)
 * tokens, parent   int32 [B][N_max]; n_nodes int32 [B] or NULL
 * err              int32 [B], REQUIRED: from tsd_tree_build_ancestors (the
 *                  walk relies on its checks)
 * u_accept, u_draw float [B][N_max], uniforms in [0, 1): u_accept[b][c] for
 *                  the test of child c, u_draw[b][i] for a draw at node i
 * next  int32 [B][N_max] out: accepted child of each node, or -1
 * draw  int32 [B][N_max] out: the drawn token of every node whose children
 *       were all rejected and of the walk's last node; -1 elsewhere (other
 *       leaves, nodes with an accepted child, padding, skipped sequences)
 * accept_len, leaf, bonus int32 [B] out; path int32 [B][D_max+1] out.
 *       A sequence with err != 0: accept_len 0, leaf -1, bonus -1, path 0.
 * workspace  >= tsd_tree_verify_stochastic_workspace_bytes() bytes: one
 *            ticket per sequence (the first 4*B bytes), ZERO-FILLED before
 *            first use and left zero-filled by every call, then per-CTA
 *            scratch that needs no initial contents.  Calls sharing one must
 *            not overlap.
 * status     int32 device word or NULL: TSD_STATUS_TIMEOUT if a bounded wait
 *            for a row copy ran out (results then unspecified).
 * No output (nor the workspace or status) may overlap an input: TSD_ERR_ARG.
 * Limits: V <= 262144 (TSD_ERR_LIMIT).
 * One launch: a cluster of up to 8 CTAs per node.  An internal node holds
 * its target row in shared memory, slice by slice, and decides its children;
 * a leaf's CTAs record per-slice sums of its target row.  The CTA that
 * finishes a sequence last walks the tree and, when the walk ends at a leaf,
 * draws the bonus token from the one slice that holds it.
 */
size_t tsd_tree_verify_stochastic_workspace_bytes(int B, int N_max, int V);
int tsd_tree_verify_stochastic(const float *logits, const float *q_draft, const int32_t *tokens,
                               const int32_t *parent, const int32_t *n_nodes, const int32_t *err,
                               const float *u_accept, const float *u_draw, int B, int N_max,
                               int V, int D_max, int32_t *next, int32_t *draw,
                               int32_t *accept_len, int32_t *leaf, int32_t *path, int32_t *bonus,
                               void *workspace, size_t ws_bytes, int32_t *status,
                               tsd_stream_t stream);
/* The launch shape tsd_tree_verify_stochastic picks on the current device:
 * CTAs per node (cluster size) and floats of the row per CTA.  Host only. */
int tsd_tree_verify_stochastic_plan(int B, int N_max, int V, int *cluster, int *slice);

/*
 * a4. Commit of the accepted path with the prefix-sharing fast reorder
 *     ([EP-zh] 2.1: path-index commit reorders the cache along the accepted
 *     path and moves only the newly accepted segment, only when needed;
 *     length-based commit is the case where nothing moves; [EP-pt] section 2).
 *
 * For k = 0..accept_len[b]: slot P_b + k receives the entry of slot
 * P_b + path[b][k] - 1, for every layer and kv head, skipped when the two are
 * equal.  All sources are read before any destination is written.
 * new_len[b] = P_b + accept_len[b] + 1; moved[b] = entries copied per
 * (layer, head).  err != 0: nothing is written, new_len = P_b, moved = 0.
 *
 * k_cache, v_cache  bf16, num_layers consecutive pools of
 *                   [num_blocks][Hkv][16][D], layer_stride elements apart.
 * block_table, prefix_len, n_nodes (or NULL: N_max nodes), accept_len, path,
 *                   err (or NULL) as produced above; path int32 [B][D_max+1].
 * new_len int32 [B] out; moved int32 [B] out or NULL; status as in a2
 * (BAD_PATH / BAD_PAGE / BAD_LEN sequences are skipped, new_len = P_b).
 */
int tsd_kv_commit_path(uint16_t *k_cache, uint16_t *v_cache, int num_layers, int64_t layer_stride,
                       const int32_t *block_table, int max_blocks, int num_blocks,
                       const int32_t *prefix_len, const int32_t *n_nodes, const int32_t *accept_len,
                       const int32_t *path, const int32_t *err, int B, int N_max, int Hkv, int D,
                       int D_max, int32_t *new_len, int32_t *moved, int32_t *status,
                       tsd_stream_t stream);

/*
 * a3 + a4 in one launch: tsd_tree_verify_greedy, and the block that finishes
 * a sequence's acceptance search then commits that sequence's accepted path
 * (every layer and kv head) exactly as tsd_kv_commit_path would from the
 * accept_len / path it has just written, which spares the commit launch.
 * Arguments: those of tsd_tree_verify_greedy (same workspace contract), then
 * those of tsd_kv_commit_path without the ones the verification produces
 * (accept_len, path) or shares (n_nodes, err, B, N_max, D_max); the tree sits
 * right after the prefix.  num_layers 0: verification only.  Outputs and
 * errors are those of the two calls; status gets the commit's BAD_PATH /
 * BAD_PAGE / BAD_LEN bits.  The fused grid writes the cache, so it does not
 * let the next kernel on the stream start before it ends (the attention pass
 * may read the cache early).  With B == 1 the one sequence's commit would run
 * in a single block: the call then launches the verification and the commit
 * kernel back to back (two launches), which measured faster.
 */
int tsd_tree_verify_greedy_commit(const float *logits, const int32_t *tokens,
                                  const int32_t *parent, const int32_t *anc, const int32_t *depth,
                                  const uint32_t *mask, const int32_t *n_nodes,
                                  const int32_t *err, int B, int N_max, int V, int D_max,
                                  int32_t *argmax, int32_t *accept_len, int32_t *leaf,
                                  int32_t *path, int32_t *bonus, void *workspace, size_t ws_bytes,
                                  uint16_t *k_cache, uint16_t *v_cache, int num_layers,
                                  int64_t layer_stride, const int32_t *block_table, int max_blocks,
                                  int num_blocks, const int32_t *prefix_len, int Hkv, int D,
                                  int32_t *new_len, int32_t *moved, int32_t *status,
                                  tsd_stream_t stream);

/*
 * a4 from a tree at its own base: as tsd_kv_commit_path, but real node i's
 * K/V are at slot tail_base[b] + i (REQUIRED, int32 [B]); slot P_b + k
 * receives the entry of slot tail_base[b] + path[b][k] - 1, the root too
 * when the two bases differ.  This materialises a deferred commit's record
 * (tail_base = the recorded tree's base).  tail_base[b] + n_nodes[b] must lie
 * inside the sequence's table (else TSD_STATUS_BAD_LEN).
 */
int tsd_kv_commit_path_from(uint16_t *k_cache, uint16_t *v_cache, int num_layers,
                            int64_t layer_stride, const int32_t *block_table, int max_blocks,
                            int num_blocks, const int32_t *prefix_len, const int32_t *n_nodes,
                            const int32_t *accept_len, const int32_t *path, const int32_t *err,
                            const int32_t *tail_base, int B, int N_max, int Hkv, int D, int D_max,
                            int32_t *new_len, int32_t *moved, int32_t *status,
                            tsd_stream_t stream);

/*
 * Deferred commit ([EP-zh] 2.1: the fast reorder moves only the accepted
 * segment, only when needed; its conclusion names commit efficiency as
 * future work).  Nothing moves: the call records where each committed entry
 * already is, and the next step's tsd_tree_attn_fwd_remap reads the committed
 * sequence through the record, with the next tree placed after the current
 * one so that no recorded entry is overwritten.  A later
 * tsd_kv_commit_path_from with the same path and tree base moves the
 * entries into place.
 *
 * prefix_len, n_nodes (or NULL), accept_len, path, err (or NULL): as
 * tsd_kv_commit_path; tail_base int32 [B] or NULL: where this step's tree
 * sits (NULL: at P_b).  Outputs, int32:
 *   remap_src  [B][D_max+1]  tail_base + path[k] - 1 for k <= accept_len,
 *                            -1 beyond (the physical slot of logical P_b + k)
 *   remap_base [B] = P_b;  remap_len [B] = accept_len + 1;
 *   new_len    [B] = P_b + accept_len + 1;
 *   next_tail  [B] = tail_base + n_nodes (where the next tree's node 0 goes).
 * A sequence with err != 0, or whose lengths or path fail the checks of
 * tsd_kv_commit_path (TSD_STATUS_BAD_LEN / BAD_PATH in *status), records
 * nothing: remap_len 0, new_len P_b, next_tail its tree base.
 * One warp per sequence.
 */
int tsd_kv_commit_remap(const int32_t *prefix_len, const int32_t *n_nodes,
                        const int32_t *accept_len, const int32_t *path, const int32_t *err,
                        const int32_t *tail_base, int B, int N_max, int D_max,
                        int32_t *remap_src, int32_t *remap_base, int32_t *remap_len,
                        int32_t *new_len, int32_t *next_tail, int32_t *status,
                        tsd_stream_t stream);

/*
 * a5. Best-first budgeted tree construction ([BASTION] Methodology 1: path
 *     score rho(i) = prod_k q_k(x_ik); Methodology 2: surrogate
 *     A_hat = sum rho, best-first expansion adds the valid node with the
 *     largest rho).
 *
 * q           float [B][K][V] per-position draft marginals (non-negative).
 * root_token  int32 [B]
 * N           node budget including the root, 1 <= N <= 256, and no larger
 *             than 1 + the number of distinct paths of length <= K.
 * parent, tokens, depth int32 [B][N] out (insertion order: parents first);
 * rho float [B][N] out, rho(child) = fl32(rho(parent) * q), rho(root) = 1;
 * ahat double [B] out, sum of rho over non-root nodes in insertion order.
 * Ties: (rho desc, depth asc, parent index asc, token rank asc); a
 * position's token rank sorts q descending, lower token id first on ties.
 * workspace  >= tsd_best_first_workspace_bytes() bytes (no initial contents).
 */
size_t tsd_best_first_workspace_bytes(int B, int K, int V, int N);
int tsd_best_first_tree_build(const float *q, const int32_t *root_token, int B, int K, int V, int N,
                              int32_t *parent, int32_t *tokens, int32_t *depth, float *rho,
                              double *ahat, void *workspace, size_t ws_bytes, tsd_stream_t stream);

/*
 * Dynamic draft trees ([Blog] EAGLE-2 section: the tree grows deep where the
 * drafter is confident and wide where it is uncertain; the page gives no
 * algorithm.  Reading: node confidence is [BASTION]'s path score, an fp32
 * product of draft probabilities along the path; expansion is level by level
 * with a frontier of the k best nodes; the N-node tree keeps the N-1 best).
 *
 * Pool (caller-owned, per sequence M_max entries): pool_parent, pool_token,
 * pool_depth int32 [B][M_max], pool_score float [B][M_max].  The root is pool
 * id 0 (parent -1, depth 0, score 1); level 1 holds ids 1..k; level l >= 2
 * holds 1 + k + (l-2) k^2 + f k + j for frontier slot f and token rank j.
 *
 * tsd_dynamic_tree_expand: one level.  Each of the F frontier nodes (F = 1 at
 * level 1 -- the root, whose entry this call writes from root_token[b] --
 * and F = k after) takes its k best tokens from its draft row q[b][f] (token
 * rank: q desc, lower id first on ties) as children with score
 * fl32(score(parent) * q); next_frontier[b] = the level's k best nodes by
 * (score desc, pool id asc).
 *   q             float [B][F][V], the drafter's distribution at each
 *                 frontier node, in frontier order (values in [0, 1]);
 *   root_token    int32 [B] (level 1 only, else ignored, may be NULL);
 *   frontier      int32 [B][F] pool ids (level >= 2; NULL at level 1): the
 *                 previous call's next_frontier;
 *   next_frontier int32 [B][k] out, must not be `frontier`.
 * Limits: 1 <= k <= 32, V >= k, the level's ids below M_max <= 8192, B <= 65535
 * (TSD_ERR_LIMIT); F other than 1 / k: TSD_ERR_ARG.  A frontier id outside
 * [0, M_max) gives children with parent -1 and score 0.
 * workspace >= tsd_dynamic_tree_workspace_bytes(B, F, k) (no initial contents).
 *
 * tsd_dynamic_tree_rerank: the root and the N-1 best of pool ids 1..M-1 by
 * (score desc, depth asc, pool id asc), in that order, into parent (re-indexed
 * to output positions; -1 for the root), tokens, depth int32 [B][N] and score
 * float [B][N].  A child never outscores its parent (q <= 1) and ranks after it,
 * so parents are kept and come first: the output is an a1-ready parent array.
 * Limits: 1 <= N <= 256, N <= M <= M_max <= 8192.
 */
size_t tsd_dynamic_tree_workspace_bytes(int B, int F, int k);
int tsd_dynamic_tree_expand(const float *q, const int32_t *root_token, int B, int F, int V, int k,
                            int level, const int32_t *frontier, int32_t *pool_parent,
                            int32_t *pool_token, int32_t *pool_depth, float *pool_score, int M_max,
                            int32_t *next_frontier, void *workspace, size_t ws_bytes,
                            tsd_stream_t stream);
int tsd_dynamic_tree_rerank(const int32_t *pool_parent, const int32_t *pool_token,
                            const int32_t *pool_depth, const float *pool_score, int B, int M,
                            int M_max, int N, int32_t *parent, int32_t *tokens, int32_t *depth,
                            float *score, tsd_stream_t stream);

/*
 * Tree budget ([BASTION] Methodology 3, hardware-aware online budget
 * controller): T_verify(N) from a roofline model of bandwidth and compute,
 * calibrated with measured step times; the tree grows until
 * S(N) = A_hat(T_N) * L_AR / C(N) starts to decrease.
 *
 * tsd_verify_step_cost (host only, no GPU work): algorithmic bytes and FLOPs
 * of one verify step (ancestor tables, attention over prefix and tree, logits,
 * at most D_max moved entries per sequence) for N-node trees, and its roofline
 * time max(bytes / BW, flops / TC) in microseconds.  prefix_len is a HOST
 * array of B lengths; hbm_gbs in GB/s, tc_tflops in TFLOP/s.  Any output
 * pointer may be NULL.  TSD_ERR_ARG on a non-positive size or peak.
 *
 * tsd_budget_calibrate (host only): least-squares line
 * t_meas ~ alpha * t_roof + beta over `count` >= 2 HOST points; TSD_ERR_ARG
 * without two distinct roofline times.
 *
 * tsd_budget_select (device, fp32 throughout): for every sequence, with A_hat(n)
 * the fp32 running sum in insertion order of rho[b][1..n-1] (the non-root
 * nodes among the first n) and S(n) = A_hat(n) * l_ar / cost[n], n_opt[b] =
 * the largest n with S(1) <= ... <= S(n) (N_max when S never decreases),
 * where S(n) < S(n-1) is tested as A_hat(n) * cost[n-1] < A_hat(n-1) * cost[n]
 * with fp32 products; s_opt[b] = fl32(fl32(A_hat(n_opt) * l_ar) / cost[n_opt]).
 *   rho    float [B][N_max] device, path scores in best-first insertion order
 *          (as tsd_best_first_tree_build writes them);
 *   cost   float [N_max + 1] device, cost[n] = C(n) = T_draft + T_verify(n)
 *          > 0 for n = 1..N_max (entry 0 unused);
 *   l_ar   > 0, the latency of one autoregressive step, in cost's unit;
 *   n_opt  int32 [B] out; s_opt float [B] out or NULL.
 * 1 <= N_max <= 256 and B <= 65535, else TSD_ERR_LIMIT.  The first n_opt[b]
 * nodes of a best-first tree form a tree (parents come first), so n_opt can
 * be passed on as n_nodes.
 */
int tsd_verify_step_cost(int B, int Hq, int Hkv, int D, const int32_t *prefix_len, int V,
                         int D_max, int N, double hbm_gbs, double tc_tflops, double *bytes,
                         double *flops, double *t_us);
int tsd_budget_calibrate(const double *t_roof, const double *t_meas, int count, double *alpha,
                         double *beta);
int tsd_budget_select(const float *rho, int B, int N_max, const float *cost, float l_ar,
                      int32_t *n_opt, float *s_opt, tsd_stream_t stream);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* TSD_H_ */
