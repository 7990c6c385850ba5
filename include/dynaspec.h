/*
 * dynaspec.h -- C ABI of the GB300 (sm_103a) DynaSpec draft head and verifier.
 *
 * DynaSpec (arXiv 2510.13847) replaces the drafter's full-vocabulary output projection with
 * a context-dependent shortlist: a small router scores vocabulary clusters from the drafter
 * hidden state, the top clusters under a position-aware budget form the shortlist V_S, the
 * head projects onto the gathered LM-head rows W[V_S] only, and the target model verifies
 * the drafted tokens over the full vocabulary by rejection sampling (abstract on
 * mlsanity.com/paper/2510.13847; summary "DynaSpec: Context-aware Dynamic Speculative
 * Sampling for Large-Vocabulary Language Models", Technical Details > Problem Definition,
 * Pipeline Flow, System Modules).  The four stages are the four calls below, in the order
 * of that pipeline:  ds_router_topk -> ds_build_shortlist -> ds_gathered_head -> ds_verify
 * (ds_verify_tree for tree drafting).
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers owned by the caller unless marked "host".  The library
 *     never allocates, frees or retains device memory.  It keeps no state between calls
 *     except in a router handle (ds_router_create: host memory the caller releases with
 *     ds_router_destroy) and the process-wide wait budget (ds_set_wait_budget).
 *   - bf16 tensors are passed as their raw 16-bit patterns (uint16_t).  Row-major layouts.
 *   - Every call is asynchronous on `stream` and returns a ds_status at once.  Errors the
 *     host can see (NULL pointers, bad sizes, a workspace that is too small, d % 8 != 0)
 *     are returned before anything is launched.  Errors only the device can see are OR-ed
 *     into *dev_status (a caller-owned int32 in device memory, which the caller zeroes and
 *     reads after synchronising); when a bit is set the outputs of that call are undefined.
 *     No call prints, exits or traps.
 *   - `ws` is caller-owned scratch of at least the size the matching *_workspace_bytes()
 *     query returns, 256-byte aligned.  Scratch that holds cross-block completion counters
 *     must be zero-filled once before its first use; each call leaves those counters at
 *     zero again.  Two calls that are in flight at the same time must not share a `ws`.
 */
#ifndef DYNASPEC_H
#define DYNASPEC_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t ds_status;

/* Host-side return codes. */
#define DS_OK               0
#define DS_ERR_INVALID_ARG  1   /* NULL pointer, size out of range, misaligned row pitch   */
#define DS_ERR_UNSUPPORTED  2   /* a size beyond what the kernels are built for            */
#define DS_ERR_CUDA         3   /* a CUDA launch or runtime call failed                     */
#define DS_ERR_WORKSPACE    4   /* ws NULL or smaller than the *_workspace_bytes() query    */

/* Device-side bits OR-ed into *dev_status. */
#define DS_DEV_BAD_INDEX    0x10  /* an id outside [0, V) or [0, M), or a draft token that is
                                     not in its shortlist                                   */
#define DS_DEV_CAPACITY     0x20  /* a shortlist larger than the capacity the caller gave   */
#define DS_DEV_TIMEOUT      0x40  /* a bounded wait inside a kernel gave up (about 1 s)     */

/* Router activations (summary, Key Hyperparameters: a two-layer MLP with ReLU activation; the
 * Tiny workload names GELU, taken in its exact erf form). */
#define DS_ACT_RELU 0
#define DS_ACT_GELU 1

/* Text for a host-side code or a device-side bit pattern.  Never NULL. */
const char *ds_status_string(ds_status s);

/* ABI version, bumped on any incompatible change. */
int ds_version(void);

/* -------------------------------------------------------------------------------------
 * ds_vocab_index -- per-token inverse of the cluster CSR.
 * The vocabulary is partitioned into M clusters (summary, Key Novelty: clusters of
 * LM-head rows), given as CSR: csr_off [M+1] (csr_off[0] = 0, csr_off[M] = V, non-
 * decreasing) and csr_tok [V] (a permutation of 0..V-1).  Fills cluster_of [V] (the
 * cluster of token v) and rank_in_cluster [V] (v's position inside its cluster's list).
 * Run once per clustering; ds_gathered_head and ds_verify look tokens up through it.
 * Device errors: DS_DEV_BAD_INDEX when a token id is outside [0, V).
 * ------------------------------------------------------------------------------------- */
ds_status ds_vocab_index(const int32_t *csr_off, const int32_t *csr_tok, int M, int V,
                         int32_t *cluster_of, int32_t *rank_in_cluster,
                         int32_t *dev_status, cudaStream_t stream);

/* -------------------------------------------------------------------------------------
 * ds_router_topk -- router MLP + position-aware top-k (summary, System Modules "Router
 * (Meta-Classifier)": a 2-layer MLP predicting relevant clusters from H_{t-1}; Key
 * Novelty and Key Hyperparameters: the budget k_c(t) shrinks with draft position t;
 * abstract: the shortlist is formed from the tokens of the best-scoring clusters).
 *   H [B, d] bf16          hidden states the router reads (H_{t-1} of each sequence)
 *   W1 [Hr, d], b1 [Hr]    first layer (out x in), bf16
 *   W2 [M, Hr], b2 [M]     second layer, bf16
 *   act                    DS_ACT_RELU or DS_ACT_GELU
 *   budget (host) [n_budget], pos (1-based draft position): k = budget[pos-1] clusters
 *   scores [B, M] fp32     out: s = W2 act(W1 h + b1) + b2 (fp32 accumulation; no sigmoid,
 *                          which would not change the top-k)
 *   cluster_ids [B, k]     out: the k highest-scoring clusters of each row, ties to the lower
 *                          id, listed in ascending id
 *   sms                    SMs to size the launches for: the ones a head running at the
 *                          same time leaves free (its free_sms).  <= 0: the default -- every
 *                          SM at pos 1 (nothing runs beside the first position's router),
 *                          else 16 at B = 1 and 8 for 2 <= B <= 64.  B > 64 ignores it.  At
 *                          B = 1 the results do not depend on it; for 2 <= B <= 64 the
 *                          fp32 summation order of the scores does (split tiles).
 * Limits: 1 <= B <= 4096, d % 8 == 0, Hr % 8 == 0, 1 <= k <= M <= 8192.
 * ws: ds_router_workspace_bytes(B, Hr) bytes (the hidden layer and completion counters:
 *     zero it once before first use).
 * ------------------------------------------------------------------------------------- */
size_t ds_router_workspace_bytes(int B, int Hr);
ds_status ds_router_topk(const uint16_t *H, int B, int d,
                         const uint16_t *W1, const uint16_t *b1, int Hr,
                         const uint16_t *W2, const uint16_t *b2, int M, int act,
                         const int32_t *budget, int n_budget, int pos,
                         float *scores, int32_t *cluster_ids, int sms,
                         void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);

/* -------------------------------------------------------------------------------------
 * Router handle -- the same router call with its weights, sizes, activation and budget table
 * bound once (summary, Problem Definition: per draft position the router's input is only the
 * hidden state H_{t-1}; the rest is fixed for the drafter).
 *   ds_router_create       checks the arguments as ds_router_topk does (plus every budget
 *                          entry in [1, M]) and returns a handle in *out.  The handle holds
 *                          non-owning views of W1, b1, W2, b2 (device memory that must outlive
 *                          it) and a host copy of budget[0..gamma).  Host memory only;
 *                          DS_ERR_UNSUPPORTED if it cannot be allocated.  *out is NULL on error.
 *   ds_router_destroy      releases the handle (NULL: no-op).  Not while a call using it is
 *                          being made on another host thread.
 *   ds_router_topk_h       ds_router_topk for draft position `pos` (1-based), sms as there.
 *                          scores may be NULL: the workspace then holds them.
 *   ds_router_workspace_bytes_h  bytes of `ws` for B hidden states (the router call's
 *                          workspace followed by room for the scores); zero it once.
 * ------------------------------------------------------------------------------------- */
typedef struct ds_router *ds_router_t;
ds_status ds_router_create(ds_router_t *out, const uint16_t *W1, const uint16_t *b1,
                           const uint16_t *W2, const uint16_t *b2, int d, int Hr, int M,
                           int act, const int32_t *budget, int gamma);
ds_status ds_router_destroy(ds_router_t r);
size_t ds_router_workspace_bytes_h(ds_router_t r, int B);
ds_status ds_router_topk_h(ds_router_t r, const uint16_t *H, int B, int pos,
                           float *scores, int32_t *cluster_ids, int sms,
                           void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);

/* -------------------------------------------------------------------------------------
 * Batch 1 without copying the list's ids.  The list of one sequence is a pure function of its
 * selected clusters and the CSR, so instead of copying the tokens (ds_build_shortlist) the
 * router's top-k block writes a table of the selected clusters, and the head reads each listed
 * token from the CSR through it: one launch fewer per draft position, same results.
 *   ds_router_topk_list_b1  ds_router_topk_h at B = 1 for draft position pos (sms as there), plus:
 *       list_table [2 (k+1)] int32 (out; 8-byte aligned): pairs {list start, CSR start} of the
 *                  k selected clusters in ascending id, then {list size, 0};
 *       cpos [M], vs_offsets [2] (out): as ds_build_shortlist writes them for one list;
 *       csr_off [M+1], V: the clusters; capacity: list entries the caller's logits hold.
 *       Device errors: DS_DEV_BAD_INDEX (a CSR slice out of range, read as empty),
 *       DS_DEV_CAPACITY (the list is longer than capacity; the table then ends the list at 0
 *       entries, so the head writes nothing).
 *       ws: ds_router_workspace_bytes_h(router, 1) bytes.
 *   ds_gathered_head_b1_table  ds_gathered_head at B = G = 1 on that list: entry j's token is
 *       csr_tok[CSR start + (j - list start)] of the last selected cluster whose list start is
 *       <= j.  k: the number of selected clusters (the table's pairs before the end pair).
 *       Outputs, free_sms and limits as ds_gathered_head's per-row path (k <= 8192);
 *       ws: ds_head_workspace_bytes(1) bytes.
 * ------------------------------------------------------------------------------------- */
ds_status ds_router_topk_list_b1(ds_router_t router, const uint16_t *H, int pos,
                                 const int32_t *csr_off, int V,
                                 float *scores, int32_t *cluster_ids,
                                 int32_t *cpos, int32_t *vs_offsets, int32_t *list_table, int64_t capacity,
                                 int sms, void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);
ds_status ds_gathered_head_b1_table(const uint16_t *H, const uint16_t *W, int V, int d,
                                    const int32_t *list_table, int k, const int32_t *csr_tok,
                                    float T, uint64_t seed, int pos,
                                    float *logits, float *row_max, float *row_sumexp,
                                    int32_t *token, int32_t *token_idx, int free_sms,
                                    void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);

/* -------------------------------------------------------------------------------------
 * ds_build_shortlist -- V_S as the union of the selected clusters (abstract; summary,
 * Problem Definition, whose output is the shortlist V_S).  Clusters partition V, so the union
 * needs no de-duplication.  Order (the pages fix only the set): selected clusters in
 * ascending id, each cluster's tokens in CSR order.
 *   cluster_ids [B, k]     ascending per row (as ds_router_topk writes them)
 *   vs_offsets [B+1]       out: list b is vs_ids[vs_offsets[b] .. vs_offsets[b+1])
 *   vs_ids [vs_capacity]   out: shortlisted token ids
 *   cpos [B, M]            out: index in list b of cluster c's first token, -1 if c is not
 *                          selected by b (ds_gathered_head and ds_verify use it)
 *   union_ids, union_cluster [V], union_count [1]: optional (all NULL or all set).  Out:
 *                          the union over the B lists of the selected clusters' tokens (same
 *                          canonical order), each token's cluster, and the union's size.
 *                          Batched and tree heads read W once over this union.
 * Device errors: DS_DEV_BAD_INDEX (cluster id outside [0, M) or not ascending),
 * DS_DEV_CAPACITY (sum of list sizes > vs_capacity; nothing past the capacity is written).
 * Limits: 1 <= B <= 4096, 1 <= k <= M <= 8192.
 * ws: ds_shortlist_workspace_bytes(B, M) bytes; holds a completion counter (zero it once;
 * every call leaves it zero).
 * ------------------------------------------------------------------------------------- */
size_t ds_shortlist_workspace_bytes(int B, int M);
ds_status ds_build_shortlist(const int32_t *csr_off, const int32_t *csr_tok, int M, int V,
                             const int32_t *cluster_ids, int B, int k,
                             int32_t *vs_offsets, int32_t *vs_ids, int64_t vs_capacity,
                             int32_t *cpos,
                             int32_t *union_ids, int32_t *union_cluster, int32_t *union_count,
                             void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);

/* -------------------------------------------------------------------------------------
 * ds_gathered_head -- logits over the shortlist only, plus the draft draw (summary, System
 * Modules "Gathered LM Head": a fused index-select + GEMM; Novel Architectural Elements
 * "Dynamic Vocabulary Head"; Key Novelty: the drafter computes logits for the dynamic
 * subset only).  W[V_S] is never materialised: rows are streamed straight from W.
 *   H [B*G, d] bf16        head rows; rows b*G .. b*G+G-1 share list b (G = 1 for chain
 *                          drafting, G = nodes per depth for tree drafting)
 *   W [V, d] bf16          the LM head
 *   vs_offsets, vs_ids, cpos, M: from ds_build_shortlist; rank_in_cluster from ds_vocab_index
 *   union_ids, union_cluster, union_count: all NULL -> each row's list is gathered on its
 *                          own (batch-1 path); all set -> W is read once over the union
 *                          of the lists and every row is scored against every union row
 *                          on the tensor cores, keeping the entries its list selects
 *   T                      temperature; 0 = greedy
 *   seed, pos              Gumbel noise key and the draft position (see below)
 *   logits (out)           row r = b*G+g writes |S_b| fp32 logits l_j = h_r . W[S_b[j]] at
 *                          logits[vs_offsets[b]*G + g*|S_b| + j]
 *   row_max, row_sumexp [B*G] (out, optional): m = max_j l_j/Te, s = sum_j exp(l_j/Te - m),
 *                          Te = T (T > 0) or 1 (T = 0)
 *   token, token_idx [B*G] (out): the draft token as a full-vocabulary id and its index j in
 *                          the list.  T = 0: argmax_j l_j.  T > 0: argmax_j (l_j/T + g_j), the
 *                          Gumbel-max draw from softmax(l/T), g_j = -log(-log u) with u from
 *                          Philox4x32-10 (key = seed, counter = (v >> 2, pos, r, 0), word v & 3,
 *                          u = (2 (w >> 9) + 1) 2^-24).  Ties go to the lower token id.  An
 *                          empty list gives token = token_idx = -1.
 *   free_sms               SMs the launch leaves free for work on other streams (the next
 *                          position's router beside the head): -1 = the default (16 on the
 *                          batch-1 per-row path, 8 on the union path, 0 otherwise); 0 = every SM
 *                          (nothing runs beside it); at least one SM is always used.
 * Limits: d % 8 == 0, d <= 16384; union path: B*G <= 128 and V <= 2^20; per-row path: G == 1
 *   and B*G <= 65535.  Larger calls return DS_ERR_UNSUPPORTED and launch nothing.
 * ws: ds_head_workspace_bytes(B*G) bytes; holds completion counters (zero it once).
 * ------------------------------------------------------------------------------------- */
size_t ds_head_workspace_bytes(int rows);
ds_status ds_gathered_head(const uint16_t *H, int B, int G,
                           const uint16_t *W, int V, int d,
                           const int32_t *vs_offsets, const int32_t *vs_ids,
                           const int32_t *cpos, int M, const int32_t *rank_in_cluster,
                           const int32_t *union_ids, const int32_t *union_cluster,
                           const int32_t *union_count,
                           float T, uint64_t seed, int pos,
                           float *logits, float *row_max, float *row_sumexp,
                           int32_t *token, int32_t *token_idx, int free_sms,
                           void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);

/* -------------------------------------------------------------------------------------
 * ds_gathered_head_noalloc -- ds_gathered_head without a workspace argument.  The DynaSpec
 * pages have no counterpart; this entry exists for callers that cannot hand the library any
 * device memory of its own: code whose device memory is owned by a pool or framework that
 * may not be grown in the middle of a step, or a plugin interface that passes only inputs
 * and outputs.  Inputs, outputs, layouts and results are those of ds_gathered_head.
 *   - Scratch is a fixed device array inside the library (about 6 MB), reserved on every
 *     GPU that loads the library until the process exits.  No call allocates or frees.
 *   - At most 32 head rows (B*G <= 32); larger calls return DS_ERR_UNSUPPORTED and launch
 *     nothing.
 *   - The first call on a device looks the array's device address up for that device
 *     (with that device current); make that first call before any stream capture.  The
 *     address is kept per device and context: after a reset of the device
 *     (cudaDeviceReset) the next call looks it up again, so that call too is a first call.
 *   - Every call shares the one array, which keeps the last call's contents; each call clears
 *     the counters it needs on `stream` before launching.  Calls that overlap on the GPU (on
 *     different streams, or from several host threads) race on the array: serialise them.
 * ------------------------------------------------------------------------------------- */
ds_status ds_gathered_head_noalloc(const uint16_t *H, int B, int G,
                                   const uint16_t *W, int V, int d,
                                   const int32_t *vs_offsets, const int32_t *vs_ids,
                                   const int32_t *cpos, int M, const int32_t *rank_in_cluster,
                                   const int32_t *union_ids, const int32_t *union_cluster,
                                   const int32_t *union_count,
                                   float T, uint64_t seed, int pos,
                                   float *logits, float *row_max, float *row_sumexp,
                                   int32_t *token, int32_t *token_idx, int free_sms,
                                   int32_t *dev_status, cudaStream_t stream);

/* -------------------------------------------------------------------------------------
 * ds_prefetch_rows -- fetch into L2 (marked evict-last) the W rows of the first `first_rows`
 * entries of the list vs_ids[offsets[0] .. offsets[1]) (offsets: two device ints, as
 * ds_build_shortlist writes them for one list).  A draft position's list is known before the
 * previous position's head has finished and its rows do not depend on that head's token, so
 * they can be fetched while that head's last rows stream; the entries a batch-1 head reads
 * first are 0 .. (its warps - 1).  A hint only: results never depend on it.  Ids outside
 * [0, V) are skipped.  blocks: 0 = 64 (the side stream's share of the GPU).
 * ------------------------------------------------------------------------------------- */
ds_status ds_prefetch_rows(const uint16_t *W, int V, int d, const int32_t *vs_ids, const int32_t *offsets,
                           int first_rows, int blocks, cudaStream_t stream);

/* -------------------------------------------------------------------------------------
 * ds_verify -- rejection-sampling verification over the full vocabulary (abstract: the target
 * model's check stays over the whole vocabulary, which keeps the output distribution exact;
 * summary, Pipeline Flow "Rejection Sampling Verification").  The pages cite Leviathan et al. and
 * Chen et al. without printing the algorithm; this is its standard statement:
 *   p_t = softmax(z_t / T) over all V, q_t = softmax(l_t / T) over the shortlist S_t (0
 *   elsewhere).  For t = 1..gamma in order accept x_t iff u_t q_t(x_t) < p_t(x_t).  At the
 *   first rejection, accepted_len = t-1 and the correction is drawn from
 *   norm(max(0, p_t - q_t)); if all gamma are accepted the bonus token is drawn from
 *   p_{gamma+1}.  Both draws are inverse-CDF in ascending token id with u_{gamma+1}; a
 *   residual without mass falls back to p_t.  T = 0: accept while x_t = argmax z_t (ties to
 *   the lower id); the correction / bonus is that argmax.
 *   p_logits [B, gamma+1, V] fp32 target logits
 *   q_logits               draft logits of position t (0-based) at q_logits + t*q_stride,
 *                          laid out as ds_gathered_head writes them with G = 1
 *   q_max, q_sumexp [gamma, B] (optional, both or neither): the draft rows' softmax
 *                          statistics as ds_gathered_head reports them (row_max, row_sumexp);
 *                          NULL -> recomputed here from q_logits
 *   vs_offsets [gamma, B+1], cpos [gamma, B*M]: the lists of each position
 *   cluster_of, rank_in_cluster [V]: from ds_vocab_index
 *   draft_ids [gamma, B]   x_t of each sequence (full-vocabulary ids)
 *   uniforms [B, gamma+1]  u_1..u_gamma for the accept tests, u_{gamma+1} for the draw
 *   accepted_len [B], correction [B] (out)
 * Device errors: DS_DEV_BAD_INDEX when a draft token is not in its shortlist.
 * Limits: 1 <= gamma <= 32, V <= 2^24, M <= 8192.
 * ws: ds_verify_workspace_bytes(B, gamma, V) bytes; holds completion counters.
 * ------------------------------------------------------------------------------------- */
size_t ds_verify_workspace_bytes(int B, int gamma, int V);
ds_status ds_verify(const float *p_logits, int B, int gamma, int V, float T,
                    const float *q_logits, int64_t q_stride,
                    const float *q_max, const float *q_sumexp,
                    const int32_t *vs_offsets, const int32_t *cpos, int M,
                    const int32_t *cluster_of, const int32_t *rank_in_cluster,
                    const int32_t *draft_ids, const float *uniforms,
                    int32_t *accepted_len, int32_t *correction,
                    void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);

/* -------------------------------------------------------------------------------------
 * ds_verify_tree -- verification of a draft tree (EAGLE-style trees, which the pages cite;
 * the pages state no tree verifier).  Reading: sibling-sequential recursive rejection, the
 * multi-draft form of speculative sampling.  Walking from the root with p = softmax(z/T) of
 * the current node, the children are tried in index order; child c is accepted iff
 * u_c q_c(x_c) < p(x_c), where q_c is c's own draft row over its depth's shortlist; after a
 * rejection p <- norm(max(0, p - q_c)) (unchanged if that has no mass).  On acceptance the
 * walk moves to c with p = softmax(z_c / T).  When no child is accepted, or at a leaf, the
 * correction is drawn from the current p by inverse CDF with u_res[depth].  T = 0: accept
 * the first child whose token is the argmax of the current node's target row.  Only the
 * target rows on the walked path are read.
 *   D depths of Wd nodes; node n = (dep-1)*Wd + i (depth-major), N = D*Wd
 *   p_logits [B, 1+N, V]   row 0: target at the root; row 1+n: target after node n
 *   parent [N] (device)    parent node of n, -1 for the root; parents sit one depth up
 *   q_logits               depth dep (0-based) at q_logits + dep*q_stride, laid out as
 *                          ds_gathered_head writes them with G = Wd
 *   q_max, q_sumexp [D, B*Wd] (optional, both or neither): the node rows' softmax statistics
 *                          as ds_gathered_head reports them; NULL -> recomputed here
 *   vs_offsets [D, B+1]    the lists of each depth; list (dep, b) holds the tokens
 *   vs_ids                 vs_ids[dep*vs_stride + vs_offsets[dep][b] + j]
 *   cpos [D, B*M], cluster_of, rank_in_cluster: as in ds_verify
 *   node_tokens [D, B*Wd]  token of node (b, dep, i) at [dep-1][b*Wd + i]
 *   u_node [B, N], u_res [B, D+1]
 *   accepted_len [B], correction [B], path [B, D] (out; accepted node ids, -1 padded)
 * Limits: D <= 32, Wd <= 64, V <= 2^24, M <= 8192.
 * ws: ds_verify_tree_workspace_bytes(B, D, Wd, V) bytes (completion counters: zero it once).
 * ------------------------------------------------------------------------------------- */
size_t ds_verify_tree_workspace_bytes(int B, int D, int Wd, int V);
ds_status ds_verify_tree(const float *p_logits, int B, int D, int Wd, int V, float T,
                         const int32_t *parent,
                         const float *q_logits, int64_t q_stride,
                         const float *q_max, const float *q_sumexp,
                         const int32_t *vs_offsets, const int32_t *vs_ids, int64_t vs_stride,
                         const int32_t *cpos, int M,
                         const int32_t *cluster_of, const int32_t *rank_in_cluster,
                         const int32_t *node_tokens, const float *u_node, const float *u_res,
                         int32_t *accepted_len, int32_t *correction, int32_t *path,
                         void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);

/* -------------------------------------------------------------------------------------
 * ds_workspace_bytes -- one query for every call's workspace (the per-call queries above give
 * the same numbers).  op and the sizes it reads:
 *   DS_OP_ROUTER       B, hidden (= Hr)                 ds_router_workspace_bytes(B, hidden)
 *   DS_OP_SHORTLIST    B, M                             ds_shortlist_workspace_bytes(B, M)
 *   DS_OP_HEAD         B, width (= G, head rows per list) ds_head_workspace_bytes(B * width)
 *   DS_OP_VERIFY       B, gamma, V                      ds_verify_workspace_bytes(B, gamma, V)
 *   DS_OP_VERIFY_TREE  B, gamma (= D), width (= Wd), V  ds_verify_tree_workspace_bytes(...)
 * Arguments an op does not read are ignored.  0 for an unknown op or sizes out of range.
 * ------------------------------------------------------------------------------------- */
#define DS_OP_ROUTER      1
#define DS_OP_SHORTLIST   2
#define DS_OP_HEAD        3
#define DS_OP_VERIFY      4
#define DS_OP_VERIFY_TREE 5
size_t ds_workspace_bytes(int op, int B, int V, int M, int gamma, int hidden, int width);

/* -------------------------------------------------------------------------------------
 * ds_set_wait_budget -- how many SM clock cycles a kernel's bounded pipeline wait (the
 * tensor-core GEMM's mbarrier waits, used by the batched router and the union head) may take
 * before it gives up and sets DS_DEV_TIMEOUT; process-wide, read when a call is made.
 * cycles = 0 restores the default (about one second at 2 GHz); cycles < 0 is refused.  Meant
 * for tests that make a wait run out on purpose (no counterpart in the method).  After a
 * call that timed out its outputs are undefined and its workspace must be zero-filled again
 * before reuse (completion counters may be left set).
 * ------------------------------------------------------------------------------------- */
ds_status ds_set_wait_budget(int64_t cycles);

/* -------------------------------------------------------------------------------------
 * Spherical k-means over the LM-head rows -- the offline step that forms the clusters the
 * router scores (summary, Key Novelty and Key Hyperparameters: the LM-head rows are clustered
 * by spherical k-means; the pages give no iteration details).  Lloyd iteration for the cosine
 * objective, centroids of unit length:
 *   ds_kmeans_init   inv_norm [V] fp32 (out): 1 / |W_v| (0 for a zero row); cent [M, d] fp32
 *                    (out): rows init_rows[0..M) of W scaled to unit length (init_rows: device,
 *                    M distinct row ids, e.g. a seeded random draw the caller makes).
 *   ds_kmeans_step   one iteration from cent (in/out):
 *                      assign [V] (out): argmax_c <W_v, bf16(cent_c)>, fp32 accumulation on the
 *                        tensor cores, ties to the lower c;
 *                      csr_off [M+1], csr_tok [V] (out): the clusters as CSR, ascending cluster
 *                        id, each cluster's tokens in ascending token id (the input of
 *                        ds_vocab_index and ds_build_shortlist);
 *                      cent (out): normalised sum of W_v * inv_norm[v] over each cluster's
 *                        tokens, added in that order in fp32; an empty cluster keeps its row.
 * Device errors: DS_DEV_BAD_INDEX for an init row outside [0, V).
 * Limits: d % 8 == 0, d <= 8192, M <= min(V, 4096), V <= 2^20.
 * ws: ds_kmeans_workspace_bytes(V, d, M) bytes (completion counters: zero it once).
 * ------------------------------------------------------------------------------------- */
size_t ds_kmeans_workspace_bytes(int V, int d, int M);
ds_status ds_kmeans_init(const uint16_t *W, int V, int d, const int32_t *init_rows, int M,
                         float *cent, float *inv_norm, int32_t *dev_status, cudaStream_t stream);
ds_status ds_kmeans_step(const uint16_t *W, int V, int d, int M, const float *inv_norm, float *cent,
                         int32_t *assign, int32_t *csr_off, int32_t *csr_tok,
                         void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);

/* -------------------------------------------------------------------------------------
 * ds_drafter_standin -- measurement helper (the drafter trunk is not part of the DynaSpec path
 * and has no trained weights here): one drafter step with the shape and weight bytes of an
 * EAGLE-style step at batch 1, so that the router's overlap with the drafter (summary, Pipeline
 * Flow; Novel Architectural Elements: the router on its own stream beside the drafter) can be
 * measured on the method's schedule.  fp32 accumulation:
 *   u = [h_prev ; E[x_prev]] (2d);  y1 = Wfc u;  y2 = Wmix y1;
 *   a_j = silu(Wug[j] . y2) * (Wug[F + j] . y2)  (j < F);  h_out = bf16(h_base + scale * (Wdn a))
 *   h_prev [d], h_base [d] bf16; x_prev (device, one int32): the previous draft token;
 *   E [V, d] bf16 (token embeddings; the LM head when they are tied);
 *   Wfc [d, 2d], Wmix [d, d], Wug [2F, d], Wdn [d, F] bf16 row-major;  h_out [d] bf16 (out).
 * h_out depends on x_prev through the whole chain; with scale = 0 it equals h_base bit for bit.
 * Device errors: DS_DEV_BAD_INDEX when x_prev is outside [0, V) (row 0 is used).
 * Limits: d % 8 == 0, F % 8 == 0.  ws: ds_drafter_standin_workspace_bytes(d, F) bytes.
 * Five launches on `stream`, on all but eight SMs (those are left to a side stream).
 * ------------------------------------------------------------------------------------- */
size_t ds_drafter_standin_workspace_bytes(int d, int F);
ds_status ds_drafter_standin(const uint16_t *h_prev, const int32_t *x_prev, int V,
                             const uint16_t *E, const uint16_t *Wfc, const uint16_t *Wmix,
                             const uint16_t *Wug, const uint16_t *Wdn, int d, int F,
                             const uint16_t *h_base, float scale, uint16_t *h_out,
                             void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);

/* -------------------------------------------------------------------------------------
 * ds_philox4x32_10 -- the device Philox4x32-10 the head draws its Gumbel noise from
 * (Salmon, Moraes, Dror, Shaw, SC'11), exposed so that it can be checked on its own.
 *   ctr [n, 4] counters, out [n, 4] words; key = the two 32-bit halves of `seed`.
 * ------------------------------------------------------------------------------------- */
ds_status ds_philox4x32_10(const uint32_t *ctr, uint64_t seed, uint32_t *out, int n,
                           cudaStream_t stream);

/* -------------------------------------------------------------------------------------
 * ds_event_record -- measurement helper (no counterpart in the method): records `event` on
 * `stream` as an external event, so that a CUDA event placed between two launches while the
 * stream is being captured into a graph becomes a real event-record node and can be timed
 * after each replay.  Outside capture it is a plain event record.
 * ------------------------------------------------------------------------------------- */
ds_status ds_event_record(cudaEvent_t event, cudaStream_t stream);

/* -------------------------------------------------------------------------------------
 * ds_copy -- transfer helper (no counterpart in the method): copies `bytes` bytes from src to
 * dst with a kernel on `stream` instead of a copy engine.  Either end may be pinned host
 * memory (page-locked, which with unified addressing the GPU reaches by its host address,
 * over NVLink-C2C on Grace systems) or device memory.  For small transfers between a step
 * and the host (hidden states in, results out) this avoids the copy engine's start-up time.
 *   dst, src               device pointers or pinned host pointers; the ranges must not
 *                          overlap.  16-byte vectors when both are 16-byte aligned and bytes %
 *                          16 == 0, else byte copies.
 * Each end is looked up with cudaPointerGetAttributes before anything is launched: device,
 * managed and page-locked host memory are accepted (page-locked memory through the device
 * alias the runtime reports); pageable or foreign host memory, which a kernel cannot reach on
 * systems without address translation services, returns DS_ERR_INVALID_ARG and launches
 * nothing.  Also DS_ERR_INVALID_ARG for NULL or overlapping ranges; bytes == 0 is a no-op.
 * ------------------------------------------------------------------------------------- */
ds_status ds_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DYNASPEC_H */
