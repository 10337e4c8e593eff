/*
 * gdn_tree.h - C ABI of the B300 (sm_103a) draft-tree verification library for
 * Gated DeltaNet (GDN) layers.
 *
 * The operation (TreeWY: Speculative Verification for Gated DeltaNet Hybrids, method and
 * novelty sections; GDN Tree-Scan abstract): given one committed recurrent state per
 * (request, head) and a parent-before-child draft tree per request, produce every draft
 * node's output as if the gated delta rule
 *
 *     S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,     o_t = S_t q_t,
 *
 * had been replayed along that node's root-to-node path (a_t = exp(g_t)), without storing a
 * state per node; then, once a path is accepted, rebuild only that path's state.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All array arguments are DEVICE pointers owned by the caller. The library allocates
 *    nothing, keeps no data between calls (gdn_tree_attention_noalloc's built-in scratch,
 *    described there, is the one exception) and never synchronises the device: each call
 *    validates its scalar arguments on the host, enqueues its kernels on `stream` and
 *    returns. Results are valid once the stream has reached that point.
 *  - Host cost: the first call on a device queries the device's properties and each kernel's
 *    shared-memory limit once; later calls reuse them (thread-safe), so an eager call costs a
 *    few microseconds of host time. A process that calls cudaDeviceReset must not call the
 *    library again afterwards (the kernels' shared-memory limits set on the old context are
 *    gone).
 *  - Layouts (T = node rows allocated, T >= cu_nodes[B]; all row-major, innermost last):
 *        ST        [B][H][d_k][d_v]  fp32   committed state S^T (S is d_v x d_k)
 *        q, k      [T][H][d_k]       bf16   (passed as uint16_t bit patterns)
 *        v         [T][H][d_v]       bf16
 *        beta, g   [T][H]            fp32   g = ln a (natural log of the gate, <= 0)
 *        parent    [T]               int32  request-local parent index, -1 = child of the
 *                                           committed state; parent[t] < t (topological order)
 *        cu_nodes  [B+1]             int32  node offsets; request r owns nodes
 *                                           cu_nodes[r] .. cu_nodes[r+1]-1 (0..64 nodes);
 *                                           non-decreasing, within [0, T]
 *        o, U      [T][H][d_v]       fp32   outputs / pseudo-values
 *        G         [T][H]            fp32   cumulative log-gate over the root-to-node path
 *        path      [B][max_path]     int32  accepted path, request-local ids, root first
 *        path_len  [B]               int32  0 = keep the committed state unchanged
 *    One tree is shared by all heads of a request; each head has its own q/k/v/beta/g.
 *  - Sizes: d_k, d_v in {32, 64, 128}; 0 <= nodes per request <= max_nodes <= 64;
 *    max_path <= 64. B may be 0 (nothing is launched). T is the number of node rows the
 *    caller allocated for q, k, v, beta, g, parent, o, U and G (T >= cu_nodes[B]); with
 *    T = 0 there are no nodes and nothing is launched.
 *  - Alignment: every array must be 16-byte aligned.
 *  - Errors: argument errors are reported by the return value before anything is launched.
 *    Data errors that only the device can see (a parent index outside [-1, t-1], a request
 *    with more than max_nodes nodes, an accepted path that is not a root-to-node chain) are
 *    OR-ed into `*status` as GDN_STATUS_* bits when `status` is non-NULL; the affected
 *    request writes nothing (no outputs, state left as it was). Kernels never trap.
 *  - Concurrency: verify only reads ST, so verifies may share a state. A commit writes ST in
 *    place and must not overlap a verify or commit of the same request on another stream.
 */
#ifndef GDN_TREE_H
#define GDN_TREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *gdn_stream_t;

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_EINVAL = 1,      /* null pointer, negative size, unsupported d_k / d_v              */
    GDN_ETOOBIG = 2,     /* max_nodes > 64, max_path > 64, or a size over a stated maximum   */
    GDN_EALIGN = 3,      /* an array is not 16-byte aligned                                  */
    GDN_ECUDA = 6,       /* a CUDA runtime call failed (no device, launch failure, ...)      */
    GDN_EARCH = 7        /* the current device cannot run sm_103a code                       */
} gdn_status;

/* Device-side data error bits, OR-ed into *status. */
#define GDN_STATUS_BAD_TREE 1u       /* parent[t] outside [-1, t-1]                          */
#define GDN_STATUS_BAD_PATH 2u       /* accepted path is not a root-to-node chain            */
#define GDN_STATUS_TOO_MANY_NODES 4u /* a request has more than max_nodes nodes              */
#define GDN_STATUS_TIMEOUT 8u        /* a bounded wait on an asynchronous copy gave up       */
#define GDN_STATUS_BAD_OFFSETS 16u   /* cu_nodes not non-decreasing inside [0, T]            */
#define GDN_STATUS_PATH_TRUNCATED 32u /* an accepted path was longer than max_path            */
#define GDN_STATUS_BAD_SLOT 64u      /* a state slot outside [0, n_slots) and not -1         */
#define GDN_STATUS_BAD_PROB 128u     /* an estimated probability outside [0, 1] or NaN        */
#define GDN_STATUS_OUT_OF_BOUNDS 256u /* debug build only: a computed index fell outside its   */
                                      /* array; that access was skipped                       */

/*
 * gdn_layout - serving layout of the *_ex entry points: how an inference engine that hosts
 * the layer (the TreeWY page evaluates it inside vLLM, experiments section) lays out its
 * recurrent states and heads. A NULL layout, or a zero-initialised one, is the plain layout
 * of gdn_tree_verify / gdn_tree_commit.
 *
 *  state_slot [B] int32 (device, or NULL): request r's state is ST[state_slot[r]] in a pool
 *             ST[n_slots][H][d_k][d_v]; -1 marks a padding request, which is skipped (no
 *             outputs, no state change); any other value outside [0, n_slots) sets
 *             GDN_STATUS_BAD_SLOT and skips the request. NULL: request r owns ST[r].
 *             Requests committed in one call must name distinct slots (verify may share).
 *  n_slots    states in the pool (> 0 when state_slot is non-NULL; ignored otherwise).
 *  H_qk       heads of q and k (0 = H). H must be a multiple of H_qk; value head h reads
 *             q/k head h / (H / H_qk) (grouped heads: consecutive value heads share a key).
 *             q and k are then [T][H_qk][d_k]; v, beta, g, o, U, G and ST keep H heads.
 *  q_scale    every query is multiplied by q_scale (o = S (q_scale q)); 0 or 1 = unscaled.
 *  a_raw, b_raw [T][H] fp32, A_log, dt_bias [H] fp32 (device; all four or none): gate fusion.
 *             With them the kernels form each node's gate and write strength themselves,
 *                 g = -exp(A_log[h]) * softplus(a_raw + dt_bias[h]),  b = sigmoid(b_raw),
 *             softplus(x) = ln(1 + e^x), sigmoid(x) = 1 / (1 + e^-x) (the gated delta rule's
 *             decay and write strength in the Gated DeltaNet parametrisation), and the beta
 *             and g arguments are not read (they may be NULL).
 */
typedef struct gdn_layout {
    const int32_t *state_slot;
    int32_t n_slots;
    int32_t H_qk;
    float q_scale;
    const float *a_raw;
    const float *b_raw;
    const float *A_log;
    const float *dt_bias;
} gdn_layout;

/*
 * gdn_tree_verify - outputs and pseudo-values of every draft node (tree-structured WY form).
 *
 * Defined by the TreeWY page (method section): pseudo-values of all candidates come from one
 * triangular system over the parent-before-child ordered tree, a node refers only to its
 * ancestors, and node outputs follow from the pseudo-values. Written out per (request, head):
 *     G_t = sum of g over t's root-to-node path,  gamma_t = exp(G_t)
 *     (I + A) U = R,   A[t,j] = b_t exp(G_t - G_j) (k_t . k_j)   for j a strict ancestor of t
 *                      R_t    = b_t (v_t - gamma_t S_0 k_t)
 *     o_t = gamma_t S_0 q_t + sum_{j ancestor of t or t itself} exp(G_t - G_j) (q_t . k_j) u_j
 * which equals the root-to-node replay of the rule (GDN Tree-Scan abstract) in exact
 * arithmetic; u_t = b_t (v_t - a_t S_parent(t) k_t) is the node's pseudo-value.
 *
 *   ST                 in   committed states, read only
 *   q, k, v, beta, g   in   node block
 *   parent, cu_nodes   in   tree shape
 *   B, H, T, d_k, d_v  in   sizes; max_nodes = an upper bound on nodes per request
 *   o, U, G            out  written for every node of every valid request
 *   status             out  optional device int32, GDN_STATUS_* bits OR-ed in
 */
gdn_status gdn_tree_verify(const float *ST, const uint16_t *q, const uint16_t *k,
                           const uint16_t *v, const float *beta, const float *g,
                           const int32_t *parent, const int32_t *cu_nodes, int32_t B, int32_t H,
                           int32_t T, int32_t d_k, int32_t d_v, int32_t max_nodes, float *o,
                           float *U, float *G, int32_t *status, gdn_stream_t stream);

/*
 * gdn_tree_verify_simt - the same operation and contract as gdn_tree_verify, computed by a
 * CUDA-core (fp32 FMA) kernel instead of the tensor-core kernel. gdn_tree_verify itself uses
 * it when d_k or d_v is 32; otherwise it serves as an in-run cross-check of the tensor-core
 * path (results agree within fp32 rounding).
 */
gdn_status gdn_tree_verify_simt(const float *ST, const uint16_t *q, const uint16_t *k,
                                const uint16_t *v, const float *beta, const float *g,
                                const int32_t *parent, const int32_t *cu_nodes, int32_t B,
                                int32_t H, int32_t T, int32_t d_k, int32_t d_v, int32_t max_nodes,
                                float *o, float *U, float *G, int32_t *status,
                                gdn_stream_t stream);

/*
 * gdn_tree_commit - rebuild the accepted path's state in place (TreeWY page, method section:
 * only the accepted path's pseudo-values are combined into the next committed state; novelty
 * section: exactly one full state is rebuilt). With l the last node of the path:
 *     ST <- exp(G_l) ST + sum_{j on the path} exp(G_l - G_j) k_j u_j^T
 * U and G are the outputs of gdn_tree_verify for the same inputs; k is its key block.
 * parent and cu_nodes are used to check that path is a root-to-node chain.
 * path_len[r] == 0 leaves request r's state untouched. Each state element is read once and
 * written once.
 */
gdn_status gdn_tree_commit(float *ST, const float *U, const float *G, const uint16_t *k,
                           const int32_t *parent, const int32_t *cu_nodes, const int32_t *path,
                           const int32_t *path_len, int32_t B, int32_t H, int32_t T,
                           int32_t d_k, int32_t d_v, int32_t max_path, int32_t *status,
                           gdn_stream_t stream);

/*
 * gdn_tree_commit_verify - gdn_tree_commit of the previous step's accepted path followed by
 * gdn_tree_verify of this step's tree, on the same state, in one pass where the shapes allow.
 *
 * In a decode loop a layer's commit for step i and its verify for step i+1 touch the same state
 * back to back. Deferring the commit to the next verify lets one kernel fold the accepted path
 * into each state row as it streams in (TreeWY page, method section: only the accepted path's
 * pseudo-values rebuild the next committed state), write the row back once and project the
 * updated row against the new tree: each state element is read once and written once for the
 * pair of operations instead of read twice. Results equal gdn_tree_commit then gdn_tree_verify.
 *
 *   ST                               in/out  committed state; updated in place
 *   U_prev, G_prev, k_prev,          in      the previous step's pseudo-values, cumulative
 *   parent_prev, cu_nodes_prev,              log-gates, keys and tree (as for gdn_tree_commit),
 *   path, path_len, T_prev, max_path         and its accepted paths
 *   q, k, v, beta, g, parent,        in      this step's tree (as for gdn_tree_verify)
 *   cu_nodes, B, H, T, d_k, d_v, max_nodes
 *   o, U, G                          out     this step's outputs; U must not alias U_prev
 *   status                           out     optional, bits of both operations
 * One fused kernel runs when d_v is 64 or 128, max_nodes <= 8 and max_path <= 4; otherwise the
 * two kernels run in order on `stream`, with the same result.
 */
gdn_status gdn_tree_commit_verify(float *ST, const float *U_prev, const float *G_prev,
                                  const uint16_t *k_prev, const int32_t *parent_prev,
                                  const int32_t *cu_nodes_prev, const int32_t *path,
                                  const int32_t *path_len, int32_t T_prev, int32_t max_path,
                                  const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                  const float *beta, const float *g, const int32_t *parent,
                                  const int32_t *cu_nodes, int32_t B, int32_t H, int32_t T,
                                  int32_t d_k, int32_t d_v, int32_t max_nodes, float *o, float *U,
                                  float *G, int32_t *status, gdn_stream_t stream);

/*
 * gdn_tree_verify_storeall - the comparison baseline the TreeWY page calls "storeall"
 * (comparison with prior methods): step every node from its parent's stored state in
 * topological order and store the state at every node.
 *     snapshots [T][H][d_k][d_v] fp32 (out): S_t^T for every node t.
 * o, U and G are produced as by gdn_tree_verify. Needs T * H * d_k * d_v * 4 bytes of
 * snapshot memory, which is what the WY form avoids.
 */
gdn_status gdn_tree_verify_storeall(const float *ST, const uint16_t *q, const uint16_t *k,
                                    const uint16_t *v, const float *beta, const float *g,
                                    const int32_t *parent, const int32_t *cu_nodes, int32_t B,
                                    int32_t H, int32_t T, int32_t d_k, int32_t d_v,
                                    int32_t max_nodes, float *snapshots, float *o, float *U,
                                    float *G, int32_t *status, gdn_stream_t stream);

/*
 * gdn_tree_commit_storeall - storeall commit: copy the stored state of the accepted path's
 * last node into ST (same path checks and path_len == 0 behaviour as gdn_tree_commit).
 */
gdn_status gdn_tree_commit_storeall(float *ST, const float *snapshots, const int32_t *parent,
                                    const int32_t *cu_nodes, const int32_t *path,
                                    const int32_t *path_len, int32_t B, int32_t H, int32_t T,
                                    int32_t d_k, int32_t d_v, int32_t max_path,
                                    int32_t *status, gdn_stream_t stream);

/*
 * gdn_tree_accept_greedy - the accepted path of every request, found on the device so that
 * verify -> accept -> commit runs without a host round trip (GDN Tree-Scan abstract: device-side
 * commitment of the accepted chain; TreeWY page, method section: candidate outputs decide
 * acceptance, after which only the accepted path's state is rebuilt).
 *
 * Greedy matching: the path starts at node 0 (the first root: the token the target already
 * produced, always kept) and, at the current node x, moves to the lowest-indexed child c with
 * draft_tok[c] == target_tok[x]; it stops when no child matches.
 *
 *   draft_tok   [T] int32   in   token proposed at each node
 *   target_tok  [T] int32   in   the target's greedy (argmax) next token after each node
 *   parent, cu_nodes        in   the tree, as for gdn_tree_verify
 *   B, T, max_nodes         in   sizes, as for gdn_tree_verify
 *   max_path                in   row length of path (>= 1 to accept anything)
 *   path     [B][max_path]  out  request-local node ids, root first; unused slots -1
 *   path_len [B]            out  0 for an empty, rejected or malformed request
 *   status                  out  optional: BAD_TREE, BAD_OFFSETS, TOO_MANY_NODES, PATH_TRUNCATED
 *                                (the path is cut at max_path nodes)
 * The outputs feed gdn_tree_commit directly.
 */
gdn_status gdn_tree_accept_greedy(const int32_t *draft_tok, const int32_t *target_tok,
                                  const int32_t *parent, const int32_t *cu_nodes, int32_t B,
                                  int32_t T, int32_t max_nodes, int32_t max_path, int32_t *path,
                                  int32_t *path_len, int32_t *status, gdn_stream_t stream);

/*
 * gdn_tree_verify_ex, gdn_tree_commit_ex, gdn_tree_commit_verify_ex - the entry points above
 * under a serving layout (gdn_layout, a HOST pointer to a struct of device pointers; NULL =
 * plain layout). Arguments, results and errors are otherwise those of gdn_tree_verify,
 * gdn_tree_commit and gdn_tree_commit_verify, with ST the state pool when state_slot is set.
 * Commit reads state_slot, n_slots and H_qk (for k) and ignores the rest. The layout fields
 * are checked on the host: H_qk < 0 or not dividing H, a non-finite q_scale, state_slot
 * without n_slots > 0, or some but not all four gate arrays give GDN_EINVAL; a misaligned
 * array gives GDN_EALIGN.
 */
gdn_status gdn_tree_verify_ex(const float *ST, const uint16_t *q, const uint16_t *k,
                              const uint16_t *v, const float *beta, const float *g,
                              const int32_t *parent, const int32_t *cu_nodes, int32_t B,
                              int32_t H, int32_t T, int32_t d_k, int32_t d_v, int32_t max_nodes,
                              const gdn_layout *layout, float *o, float *U, float *G,
                              int32_t *status, gdn_stream_t stream);

gdn_status gdn_tree_commit_ex(float *ST, const float *U, const float *G, const uint16_t *k,
                              const int32_t *parent, const int32_t *cu_nodes, const int32_t *path,
                              const int32_t *path_len, int32_t B, int32_t H, int32_t T,
                              int32_t d_k, int32_t d_v, int32_t max_path, const gdn_layout *layout,
                              int32_t *status, gdn_stream_t stream);

/* The previous step's requests and this step's are the same requests in the same order; both
 * use layout->state_slot, and k_prev has H_qk heads like k. q_scale and the gate arrays belong
 * to this step's tree (the previous step's gates are already folded into G_prev). */
gdn_status gdn_tree_commit_verify_ex(float *ST, const float *U_prev, const float *G_prev,
                                     const uint16_t *k_prev, const int32_t *parent_prev,
                                     const int32_t *cu_nodes_prev, const int32_t *path,
                                     const int32_t *path_len, int32_t T_prev, int32_t max_path,
                                     const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                     const float *beta, const float *g, const int32_t *parent,
                                     const int32_t *cu_nodes, int32_t B, int32_t H, int32_t T,
                                     int32_t d_k, int32_t d_v, int32_t max_nodes,
                                     const gdn_layout *layout, float *o, float *U, float *G,
                                     int32_t *status, gdn_stream_t stream);

/*
 * gdn_tree_budget_topb - adaptive verification budget (DSpark adaptive-verification news item:
 * each draft token's estimated probability of passing verification gives, per request, the
 * probability that its sequence survives to each position; one global budget B goes to the
 * positions with the largest survival probabilities across all requests).
 *
 *   p_accept  [R][K] fp32  in   estimated acceptance probability of draft position i of
 *                               request r; values outside [0, 1] or NaN count as 0 and set
 *                               GDN_STATUS_BAD_PROB
 *   R, K, budget           in   requests, draft positions per request (1..63), positions to
 *                               verify in total (>= 0); R * K <= 16384 and 12 R K + 4 R
 *                               <= 232448 (one CTA's shared memory), else GDN_ETOOBIG
 *   n_sel     [R]    out        positions chosen for request r - always its first n_sel[r]
 *   survival  [R][K] out        optional: s[r][i] = p[r][0] * ... * p[r][i] (fp32, in that order)
 *   cu_nodes  [R+1]  out        optional: the verify batch, one chain per request of 1 + n_sel[r]
 *                               nodes (the token the target already produced, then the drafts)
 *   parent    [R + min(budget, R K)] out   optional (needs cu_nodes): the chains' parents
 * Order: survival descending, equal values by (request, position) ascending; the choice is
 * exact (fp32 products, compared as numbers). One CTA; the result is a function of the inputs.
 */
gdn_status gdn_tree_budget_topb(const float *p_accept, int32_t R, int32_t K, int32_t budget,
                                int32_t *n_sel, float *survival, int32_t *cu_nodes,
                                int32_t *parent, int32_t *status, gdn_stream_t stream);

/*
 * gdn_tree_grow_best_first - threshold best-first draft-tree growth (TreeSpark page: the tree
 * grows along its most promising branch first and stops when the value of the best remaining
 * candidate drops below a threshold; a candidate's value is the survival product along its
 * branch).
 *
 * Candidates per request form a complete fanout-ary tree of the given depth, numbered
 * breadth-first: 0 is the root (the token the target already produced, value 1, always
 * taken), the children of c are fanout*c + 1 .. fanout*c + fanout, C = sum_l fanout^l <= 8192.
 *   p_edge [R][C] fp32  in   estimated probability that candidate c is accepted given its
 *                            parent (column 0 unused); invalid values count as 0 (BAD_PROB)
 *   threshold           in   a candidate is taken while its value >= threshold
 *   max_nodes           in   at most this many nodes per request (0..64)
 *   n_nodes      [R]              out  nodes taken per request
 *   parent_local [R][max_nodes]   out  request-local parent of each taken node, in the order
 *                                      taken (parent before child), -1 for the root and past n
 *   cand, value  [R][max_nodes]   out  optional: candidate index and value of each taken node
 *                                      (-1 / 0 past n)
 *   cu_nodes [R+1], parent [R * max_nodes]   out  optional (both or neither): the same trees
 *                                      packed as a ragged verify batch
 * The order taken is value descending, equal values by candidate index ascending, which is
 * the best-first order because values never grow along a branch.
 */
gdn_status gdn_tree_grow_best_first(const float *p_edge, int32_t R, int32_t fanout, int32_t depth,
                                    float threshold, int32_t max_nodes, int32_t *n_nodes,
                                    int32_t *parent_local, int32_t *cand, float *value,
                                    int32_t *cu_nodes, int32_t *parent, int32_t *status,
                                    gdn_stream_t stream);

/*
 * gdn_tree_attention - tree-bias attention for the attention layers of a hybrid model (GDN
 * Tree-Scan abstract: tree-bias attention beside the recurrent-state replay; an attention-only
 * verifier mainly needs the ancestry mask). Draft node t of request r, query head h (key/value
 * head h / (H_q / H_kv)), attends to every key of the request's committed prefix and to the
 * draft nodes on its own root-to-node path, itself included:
 *     o[t][h] = sum_j softmax_j(scale * q[t][h] . k_j) v_j   over those keys j
 *
 *   q        [T][H_q][d]        bf16  in   the draft nodes' queries
 *   k, v     [T][H_kv][d]       bf16  in   the draft nodes' own keys and values
 *   k_cache, v_cache [P_total][H_kv][d] bf16 in   committed prefixes; request r owns rows
 *                                          cu_prefix[r] .. cu_prefix[r+1]-1 (may be NULL when
 *                                          P_total is 0)
 *   cu_prefix [B+1], parent [T], cu_nodes [B+1] int32 in   as for gdn_tree_verify; at most
 *                                          max_nodes (<= 64) nodes and max_prefix keys per request
 *   d                                 64 or 128; H_q / H_kv a power of two <= 128
 *   scale                             score scale, > 0 (e.g. d^-1/2)
 *   o        [T][H_q][d]        fp32  out  written for every node of every valid request
 *   workspace, workspace_bytes        optional device scratch: where the (request, head, query
 *                                     tile) grid fills the GPU's SMs poorly (one CTA per SM: too
 *                                     few CTAs, or a thin last wave), long prefixes are split
 *                                     across CTAs and merged, using up to
 *                                     gdn_tree_attention_workspace_size() bytes of it; with NULL
 *                                     or less, fewer splits (none) are made
 *   status                            optional: BAD_OFFSETS (offsets outside T / P_total, or a
 *                                     prefix longer than max_prefix), TOO_MANY_NODES, BAD_TREE,
 *                                     TIMEOUT; the request then writes nothing
 * Scores and the running softmax are fp32; the probabilities enter P.V rounded to bf16 (the
 * tensor-core operand type), so |o - o_exact| <= 2^-8 max|v| per output.
 */
gdn_status gdn_tree_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                              const uint16_t *k_cache, const uint16_t *v_cache,
                              const int32_t *cu_prefix, const int32_t *parent,
                              const int32_t *cu_nodes, int32_t B, int32_t H_q, int32_t H_kv,
                              int32_t T, int32_t P_total, int32_t d, int32_t max_nodes,
                              int32_t max_prefix, float scale, float *o, void *workspace,
                              size_t workspace_bytes, int32_t *status, gdn_stream_t stream);

/* Workspace bytes gdn_tree_attention uses at most for these sizes on the current device (0 when
 * it would not split). */
size_t gdn_tree_attention_workspace_size(int32_t B, int32_t H_q, int32_t H_kv, int32_t d,
                                         int32_t max_nodes, int32_t max_prefix);

/*
 * gdn_tree_attention_noalloc - gdn_tree_attention for callers that cannot allocate device
 * memory: a serving engine whose allocator reserved the GPU's memory at start-up for its KV-cache
 * pool, or a host framework that forbids allocation inside a forward step, has no buffer to
 * offer as workspace. The pages have no counterpart of this entry point; it only moves the
 * workspace of the key splits into scratch the library owns.
 *
 * Same arguments and results as gdn_tree_attention, without workspace and workspace_bytes. Its
 * key splits live in a 32 MiB scratch array built into the library. It makes the splits that
 * gdn_tree_attention makes with a 32 MiB workspace: the same plan (and bit-identical results) as
 * with gdn_tree_attention_workspace_size() bytes whenever that is at most 32 MiB, otherwise
 * fewer splits (at worst none, which needs no scratch), so every valid size runs. A plan larger
 * than the scratch cannot occur; the entry point would return GDN_ETOOBIG with a message on
 * stderr before launching anything. It calls no allocator.
 *
 * The array is device memory of the library's module: the driver reserves it on a device when
 * the module is first loaded there (under CUDA's default lazy loading, at the library's first
 * use on that device), and keeps it until the process exits. The first call that needs scratch
 * on a device also looks up the array's device address there and keeps it. So make a first call
 * on each device before reserving the rest of its memory for a pool, and before any stream
 * capture; after cudaDeviceReset the kept address is stale and this entry point must not be
 * used again in that process. Every call shares the one array and writes the parts it reads,
 * so nothing needs clearing between calls, but two calls that overlap on the GPU (other
 * streams, other host threads) race on it.
 */
gdn_status gdn_tree_attention_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                      const uint16_t *k_cache, const uint16_t *v_cache,
                                      const int32_t *cu_prefix, const int32_t *parent,
                                      const int32_t *cu_nodes, int32_t B, int32_t H_q, int32_t H_kv,
                                      int32_t T, int32_t P_total, int32_t d, int32_t max_nodes,
                                      int32_t max_prefix, float scale, float *o, int32_t *status,
                                      gdn_stream_t stream);

/* Human-readable name of a return code (static string, never NULL). */
const char *gdn_status_str(gdn_status s);

/* ABI version of this header (incremented on incompatible changes). */
int32_t gdn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_TREE_H */
