/*
 * medusa.h -- C ABI of the B300 (sm_103a) Medusa decode-step library.
 *
 * One Medusa decode step, as the method is described on the source pages
 * (Ultralytics glossary "Medusa Heads"; wiblog.cn "Medusa multi-head
 * speculative decoding"; cnnetsun.cn "Medusa safety considerations";
 * jisaku.com glossary "Medusa (LLM decoding)"):
 *
 *   medusa_heads_topk     K Medusa heads h + SiLU(W1 h + b1) -> W2, per-head top-k
 *   medusa_build_tree     per-head top-k -> tokens / position ids of a fixed candidate tree
 *   medusa_tree_attention one tree-masked attention pass over KV cache + tree
 *   medusa_verify_accept  lm_head logits of every tree node + typical acceptance
 *   medusa_kv_commit      accepted path's K/V rows appended to the cache
 *
 * Conventions shared by every call
 *   - Tensor pointers are DEVICE pointers owned by the caller; the library
 *     never frees or keeps them.  Pointers to host arrays are named *_host.
 *   - Every device pointer must be 16-byte aligned (MEDUSA_ERR_ALIGNMENT).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Per-step calls allocate nothing, copy nothing to or
 *     from the host and never synchronise, so a whole step can be captured
 *     in a CUDA graph.  Scratch memory is the caller's `ws` buffer of at
 *     least the size the matching *_workspace_size() returns; it must be
 *     zero-filled once before its first use and is left ready for the next
 *     call (self-resetting counters).  Two calls in flight at the same time
 *     must not share one workspace.
 *   - Layouts are row-major, innermost dimension last, nn.Linear weights
 *     [out, in].  Floating-point tensors are all of one `medusa_dtype`
 *     (fp32 or bf16); accumulations are fp32; every float output is fp32.
 *   - Return value: MEDUSA_OK (0) or a negative medusa_status detected on
 *     the host before anything was launched (MEDUSA_ERR_CUDA: a launch or
 *     a CUDA call failed).  Conditions found on the device are OR-ed into
 *     the caller's int32 dev_status[B] (MEDUSA_DEV_* bits; the caller zeroes
 *     it); no kernel traps or asserts.
 *   - Tree-indexed tensors use the tree's canonical node order: the root,
 *     then nodes by depth, then by rank tuple.
 *   - Kernels are launched with programmatic dependent launch: a call may
 *     start while the previous kernel on the stream is still finishing, and
 *     waits for it before reading anything that work could have produced.
 *     The weights (w1, b1, w2, lm_head) are treated as constant inputs of the
 *     step and may be streamed before that wait, so a caller that rewrites
 *     weights on the same stream must complete that write first (an event
 *     wait or a stream synchronisation between the write and the call).
 */
#ifndef MEDUSA_H_
#define MEDUSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* medusa_stream_t; /* same type as cudaStream_t */

typedef enum {
  MEDUSA_OK = 0,
  MEDUSA_ERR_INVALID_ARG = -1, /* null pointer, size out of range, bad tree spec */
  MEDUSA_ERR_ALIGNMENT = -2,   /* a device pointer is not 16-byte aligned      */
  MEDUSA_ERR_UNSUPPORTED = -3, /* shape outside what the kernels implement      */
  MEDUSA_ERR_WORKSPACE = -4,   /* ws missing or smaller than *_workspace_size   */
  MEDUSA_ERR_CUDA = -5,        /* a CUDA call or kernel launch failed           */
  MEDUSA_ERR_SCRATCH_LIMIT = -6 /* shape needs more than the built-in scratch   */
} medusa_status;

/* bits OR-ed into dev_status[b] */
#define MEDUSA_DEV_KV_OVERFLOW 1 /* kv_len + accepted rows would pass Lmax: cache left untouched */
#define MEDUSA_DEV_NAN 2         /* a NaN logit or statistic was met                           */
#define MEDUSA_DEV_TIMEOUT 4     /* a bounded device wait gave up (result of that launch invalid) */
#define MEDUSA_DEV_BAD_TOKEN 8   /* a tree node got no candidate (top-k entry missing)          */

typedef enum { MEDUSA_F32 = 0, MEDUSA_BF16 = 1 } medusa_dtype;

#define MEDUSA_MAX_DEPTH 16   /* deepest tree node            */
#define MEDUSA_MAX_NODES 4096 /* T = candidate nodes + root   */
#define MEDUSA_MAX_BATCH 64
#define MEDUSA_MAX_TOPK 64

const char* medusa_status_string(int status);

/* Number of kernels this library has launched (or recorded into a stream
 * capture) in this process so far; a diagnostic for counting launches. */
uint64_t medusa_kernel_launches(void);

/* ------------------------------------------------------------------------
 * Candidate tree ("medusa_choices").
 * A fixed tree is given as a list of rank tuples: choice (r1..rd) is the
 * node whose depth-j token is head j's rank-rj candidate; its parent is the
 * tuple without the last rank.  The tree is regular and fixed, so its
 * tables (parents, depths, ancestor mask, paths) are built once here and
 * cached on the device (wiblog "Tree attention"; Ultralytics "Tree
 * attention and accepting tokens"; cnnetsun "Key safety parameters",
 * medusa_choices).
 *   ranks_flat_host: all tuples concatenated; lens_host[n_choices]: their lengths.
 *   The list must be prefix-closed and free of duplicates, ranks >= 0,
 *   depth <= MEDUSA_MAX_DEPTH, 1 + n_choices <= MEDUSA_MAX_NODES
 *   (MEDUSA_ERR_INVALID_ARG otherwise).  The device tables live on the
 *   device current at the call; this call allocates and copies synchronously.
 * ---------------------------------------------------------------------- */
typedef struct medusa_tree medusa_tree;

typedef struct {
  int32_t T;                          /* nodes incl. root                        */
  int32_t P;                          /* paths = leaves                          */
  int32_t dmax;                       /* deepest node's depth                    */
  int32_t mask_words;                 /* u32 words per ancestor-mask row         */
  int32_t max_rank[MEDUSA_MAX_DEPTH]; /* largest rank used at depth d+1          */
} medusa_tree_info;

int medusa_tree_create(const int32_t* ranks_flat_host, const int32_t* lens_host,
                       int32_t n_choices, medusa_tree** out);
int medusa_tree_get_info(const medusa_tree* tree, medusa_tree_info* info);
/* The tree's sizes one by one (any pointer may be NULL): T nodes including the
 * root, P paths, dmax, and topk_per_depth[MEDUSA_MAX_DEPTH]: entry d is the
 * number of top-k candidates head d+1 must supply (largest rank used at depth
 * d+1, plus one; 0 past dmax). */
int medusa_tree_query(const medusa_tree* tree, int32_t* T, int32_t* P, int32_t* dmax,
                      int32_t* topk_per_depth);
/* Host copies of the tables (any pointer may be NULL): parent[T] (-1 root),
 * depth[T], rank[T] (-1 root), mask[T * mask_words] (bit j of row i set iff
 * node j is i or an ancestor of i), paths[P * (dmax+1)] (node ids root->leaf,
 * -1 padded, leaves in canonical order). */
int medusa_tree_copy_tables(const medusa_tree* tree, int32_t* parent_host, int32_t* depth_host,
                            int32_t* rank_host, uint32_t* mask_host, int32_t* paths_host);
void medusa_tree_destroy(medusa_tree* tree);

/* ------------------------------------------------------------------------
 * medusa_heads_topk
 * Head k on the last hidden state h: u_k = h + SiLU(W1_k h + b1_k), logits
 * z_k = W2_k u_k; each head keeps its top-k tokens (Ultralytics "How the
 * heads predict the next tokens": one FC layer with SiLU and a residual,
 * then a bias-free vocabulary projection; wiblog "Medusa decoding heads":
 * each head outputs its top-k candidates).
 *   h [B,H]; w1 [K,H,H]; b1 [K,H]; w2 [K,V,H]; lm_head [V,H] or NULL.
 *   head_logits [B,K,V] fp32 or NULL.
 *   topk_ids [B,K,topk] int32, topk_vals [B,K,topk] fp32: descending, ties to
 *     the lower token id; NaN logits rank below every number.
 *   root_tok [B] int32: if lm_head != NULL it receives argmax lm_head(h) (the
 *     base model's greedy next token, ties to the lower id); otherwise it is
 *     not touched (it then holds the previous step's next_root).
 *   For bf16 data u is rounded to bf16 before W2 (the W2 stream is bf16).
 *   Limits: 1 <= B <= MEDUSA_MAX_BATCH, H % 8 == 0, 1 <= topk <= min(V, MEDUSA_MAX_TOPK).
 *   A row with fewer than topk numbers among its logits (NaN logits) gets id
 *   -1 and value -inf in the entries left over.
 *   bf16 with B >= 3 and lm_head == NULL runs W1 h and W2_k u_k on the tensor
 *   cores; the workspace then also holds the [B,K*H] fp32 first-layer outputs
 *   and, with topk <= 16, the top-k candidates each vocabulary tile of the W2
 *   GEMM keeps in its epilogue (a [B,K,tiles,topk] value/id pair, merged per
 *   row and head by a second launch), else the [B,K,V] fp32 logits
 *   (medusa_heads_topk_workspace_size includes them).
 * ---------------------------------------------------------------------- */
size_t medusa_heads_topk_workspace_size(int32_t B, int32_t H, int32_t V, int32_t K, int32_t topk,
                                        int32_t with_lm_head, medusa_dtype dtype);
int medusa_heads_topk(const void* h, const void* w1, const void* b1, const void* w2,
                      const void* lm_head, int32_t B, int32_t H, int32_t V, int32_t K,
                      int32_t topk, medusa_dtype dtype, float* head_logits, int32_t* topk_ids,
                      float* topk_vals, int32_t* root_tok, void* ws, size_t ws_bytes,
                      medusa_stream_t stream);

/* ------------------------------------------------------------------------
 * medusa_heads_topk_tree
 * The Medusa heads on the tree nodes' hidden states, of which each request
 * keeps the top-k of its accepted node: the candidates of the next step come
 * out of the verification pass with no separate pass over the accepted token
 * (wiblog "Inference flow in an online chat service"; the accepted branch
 * continues the sequence, Ultralytics "Tree attention and accepting
 * tokens").  For node row x[b,i]: u_k = x + SiLU(W1_k x + b1_k), z_k = W2_k u_k;
 * request b keeps the top-k of row best_node[b].  Acceptance is known when
 * this runs, so the accepted rows are gathered first and the heads run on
 * those B rows (bf16 with B >= 3: both head products as tcgen05 GEMMs), which
 * gives the same outputs as running them on every node.
 *   x [B,T,H] (the tree nodes' hidden states, as given to
 *   medusa_verify_accept); w1, b1, w2 as in medusa_heads_topk;
 *   best_node [B] int32 device (medusa_verify_accept's output; values outside
 *   [0, T) are clamped).
 *   head_logits [B,K,V] fp32 or NULL: the logits of the accepted rows.
 *   topk_ids, topk_vals [B,K,topk]: as medusa_heads_topk, ready for the next
 *   step's medusa_build_tree together with medusa_verify_accept's next_root.
 *   Limits as medusa_heads_topk.  The workspace holds the gathered [B,H] rows
 *   and medusa_heads_topk's workspace for B rows without lm_head.
 * ---------------------------------------------------------------------- */
size_t medusa_heads_topk_tree_workspace_size(const medusa_tree* tree, int32_t B, int32_t H, int32_t V,
                                             int32_t K, int32_t topk, medusa_dtype dtype);
int medusa_heads_topk_tree(const medusa_tree* tree, const void* x, const void* w1, const void* b1,
                           const void* w2, const int32_t* best_node, int32_t B, int32_t H, int32_t V,
                           int32_t K, int32_t topk, medusa_dtype dtype, float* head_logits,
                           int32_t* topk_ids, float* topk_vals, void* ws, size_t ws_bytes,
                           medusa_stream_t stream);

/* ------------------------------------------------------------------------
 * medusa_heads_topk_noalloc
 * No counterpart on the source pages: a convenience of this library.
 * The computation, arguments and outputs of medusa_heads_topk, minus the
 * workspace, for callers that cannot allocate device memory: cudaMalloc may
 * synchronise the device and takes a driver-wide lock, so latency-bound decode
 * loops, plugins living inside another framework's memory pool and programs
 * with a fixed device-memory budget often may not call it.  The scratch is a
 * fixed array of MEDUSA_NOALLOC_SCRATCH_BYTES compiled into the library; every
 * GPU that loads the library holds it until the process exits.
 *   - Always the CUDA-core path (heads_fc + heads_vocab): it never takes the
 *     tensor-core path that medusa_heads_topk uses for bf16 with B >= 3 and no
 *     lm_head, so in that case results can differ from medusa_heads_topk at
 *     near-ties (both match the exact heads within the float tolerance) and the
 *     call streams the weights on CUDA cores.
 *   - Shapes whose scratch would exceed the array return
 *     MEDUSA_ERR_SCRATCH_LIMIT.  The scratch a shape needs is what
 *     medusa_heads_topk_workspace_size returns for the same arguments whenever
 *     that plan is also the CUDA-core one (fp32, B <= 2, or lm_head given; e.g.
 *     the Llama-8B shape at batch 16 with lm_head needs about 1.5 MB).
 *   - The array's device address is looked up on every call made outside a
 *     stream capture; the first call on each device (and the first after a
 *     device reset) must come before any stream capture on that device, since
 *     it also loads the library's device code.  A call inside a capture reuses
 *     the address found by the last call outside one.
 *   - All calls share the one array and it keeps the last call's contents;
 *     the ticket counters are cleared on the stream at every call.  Calls
 *     that overlap on the GPU (other streams, other host threads) race.
 *   - Allocates nothing: no cudaMalloc/cudaFree, no allocating library routine.
 * ---------------------------------------------------------------------- */
#define MEDUSA_NOALLOC_SCRATCH_BYTES (8u << 20)
int medusa_heads_topk_noalloc(const void* h, const void* w1, const void* b1, const void* w2,
                              const void* lm_head, int32_t B, int32_t H, int32_t V, int32_t K,
                              int32_t topk, medusa_dtype dtype, float* head_logits, int32_t* topk_ids,
                              float* topk_vals, int32_t* root_tok, medusa_stream_t stream);

/* ------------------------------------------------------------------------
 * medusa_build_tree
 * Token and position id of every tree node: the root token at depth 0, head
 * d's rank-r candidate for a depth-d node of rank r -- the same head-d tokens
 * under every branch (Ultralytics "Tree attention and accepting tokens");
 * position = kv_len[b] + depth (wiblog "Tree attention": every token gets
 * its correct position index).
 *   root_tok [B]; topk_ids [B,K,topk] (from medusa_heads_topk); kv_len [B].
 *   tree_tokens [B,T], position_ids [B,T] int32 out.
 *   candidates [B,P,dmax+1] int32 out or NULL: token sequence of each path, -1 padded.
 *   Requires tree dmax <= K and every rank < topk (MEDUSA_ERR_INVALID_ARG).
 *   A node whose candidate id is negative sets MEDUSA_DEV_BAD_TOKEN.
 * ---------------------------------------------------------------------- */
int medusa_build_tree(const medusa_tree* tree, const int32_t* root_tok, const int32_t* topk_ids,
                      int32_t B, int32_t K, int32_t topk, const int32_t* kv_len,
                      int32_t* tree_tokens, int32_t* position_ids, int32_t* candidates,
                      int32_t* dev_status, medusa_stream_t stream);

/* ------------------------------------------------------------------------
 * medusa_tree_attention
 * One attention pass of all tree tokens over the KV cache plus the tree:
 * node i attends to the kv_len[b] cached keys and to the tree keys of its
 * ancestors and itself only (wiblog "Tree attention": each token may attend
 * only to the tokens on its own prefix path, every token with its correct
 * position index; Ultralytics "Tree attention and accepting tokens").
 * o = softmax(scale * q k^T) v.
 *   q [B,T,Hq,D]; k_new, v_new [B,T,Hkv,D]; k_cache, v_cache [B,Hkv,Lmax,D];
 *   kv_len [B] device, each in [0, Lmax]; out [B,T,Hq,D] fp32.
 *   Query head hq reads key/value head hq / (Hq/Hkv) (grouped-query attention).
 *   Position encoding (no counterpart on the pages beyond "correct position
 *   index"; rotary embedding as in Su et al., "RoFormer", 2021):
 *     rope == 0: q and k_new are taken as given, already position-encoded
 *       (the layer that produces them is outside this library);
 *       position_ids is unused and may be NULL.
 *     rope != 0: q and k_new are first rotated at position_ids [B,T] int32
 *       (device; medusa_build_tree's output, kv_len + depth), rotate-half
 *       form: for d < D/2 the pair (x[d], x[d+D/2]) turns by
 *       position * rope_theta^(-2d/D) (rope_theta > 1, e.g. 10000).  The cache
 *       keys are taken as already rotated at their own positions.  When k_rot
 *       is not NULL the rotated keys [B,T,Hkv,D] (dtype) are written there, so
 *       that medusa_kv_commit can append rotated keys to the cache; otherwise
 *       they stay in the workspace.
 *   kv_len_hint: host upper bound of kv_len (0 = Lmax); used only to size the
 *   split of the cache across CTAs, any kv_len <= Lmax is handled.
 *   Limits: D in {64, 128}; Hq % Hkv == 0; Hq <= 128.
 *   After MEDUSA_DEV_TIMEOUT the workspace must be zero-filled again.
 * ---------------------------------------------------------------------- */
size_t medusa_tree_attention_workspace_size(const medusa_tree* tree, int32_t B, int32_t Hq,
                                            int32_t Hkv, int32_t D, int32_t Lmax,
                                            int32_t kv_len_hint, medusa_dtype dtype);
int medusa_tree_attention(const medusa_tree* tree, const void* q, const void* k_new,
                          const void* v_new, const void* k_cache, const void* v_cache,
                          const int32_t* kv_len, const int32_t* position_ids, int32_t B, int32_t Hq,
                          int32_t Hkv, int32_t D, int32_t Lmax, int32_t kv_len_hint, float scale,
                          int32_t rope, float rope_theta, medusa_dtype dtype, float* out, void* k_rot,
                          void* ws, size_t ws_bytes, int32_t* dev_status, medusa_stream_t stream);

/* ------------------------------------------------------------------------
 * medusa_verify_accept
 * lm_head logits of every tree node, z[b,i] = lm_head . x[b,i] (wiblog
 * "Inference flow": the original model computes every candidate's
 * probability in one verification pass), then typical acceptance (wiblog
 * "Typical acceptance"; cnnetsun "Posterior probability evaluation",
 * evaluate_posterior -> best_candidate, accept_length):
 *   temperature == 0: node c is accepted iff its token is argmax z[parent(c)]
 *     (ties to the lower id);
 *   temperature  > 0: q = softmax(z[parent(c)] / temperature), p = q[token(c)],
 *     H = -sum q ln q; accepted iff p > min(posterior_threshold,
 *     posterior_alpha * exp(-H)).
 *   A node is kept iff it is accepted and its parent is kept; the root is
 *   always kept (the first token is the greedy one).  The deepest kept node
 *   wins; among equally deep kept nodes (the pages leave the choice open):
 *     tie_break 0: the first in canonical order (higher-ranked candidates);
 *     tie_break 1: the one whose path has the highest joint probability (the
 *       product of each node's p under its parent), equal products to the
 *       first in canonical order (at temperature 0 every kept p is 1).
 * Outputs (device):
 *   logits [B,T,V] fp32 or NULL; node_p [B,T] or NULL (p of node c under its
 *   parent; 1/0 = match/miss at temperature 0; 1 for the root); node_H [B,T]
 *   or NULL (entropy of node i's own tempered distribution; 0 at temperature 0);
 *   accept_len [B] (depth of the winner = tokens accepted beyond the root);
 *   best_node [B]; best_path [B] (first path through the winner);
 *   accepted_tokens [B, dmax+1] (root..winner, -1 padded);
 *   next_root [B] (argmax of the winner's logits).
 *   Requires x [B,T,H]; tree_tokens [B,T] from medusa_build_tree; temperature
 *   >= 0; H % 8 == 0.
 * ---------------------------------------------------------------------- */
size_t medusa_verify_accept_workspace_size(const medusa_tree* tree, int32_t B, int32_t H,
                                           int32_t V, medusa_dtype dtype);
int medusa_verify_accept(const medusa_tree* tree, const void* x, const void* lm_head,
                         const int32_t* tree_tokens, int32_t B, int32_t H, int32_t V,
                         medusa_dtype dtype, float temperature, float posterior_threshold,
                         float posterior_alpha, int32_t tie_break, float* logits, float* node_p, float* node_H,
                         int32_t* accept_len, int32_t* best_path, int32_t* best_node,
                         int32_t* accepted_tokens, int32_t* next_root, int32_t* dev_status,
                         void* ws, size_t ws_bytes, medusa_stream_t stream);

/* ------------------------------------------------------------------------
 * medusa_verify_accept_commit
 * medusa_verify_accept followed by medusa_kv_commit of its winner, with one
 * launch fewer: the CTA that runs a request's acceptance also copies the
 * accepted path's K/V rows (depth 0..accept_len) from k_new/v_new into the
 * cache at kv_len.. and advances kv_len, with medusa_kv_commit's rules (a
 * request whose rows would pass Lmax is flagged MEDUSA_DEV_KV_OVERFLOW and
 * left untouched).  Arguments as the two calls; k_new, v_new [B,T,Hkv,D] and
 * the cache [B,Hkv,Lmax,D] in `dtype`; (D * element size) % 16 == 0.  The
 * workspace is medusa_verify_accept's.
 * ---------------------------------------------------------------------- */
int medusa_verify_accept_commit(const medusa_tree* tree, const void* x, const void* lm_head,
                                const int32_t* tree_tokens, int32_t B, int32_t H, int32_t V,
                                medusa_dtype dtype, float temperature, float posterior_threshold,
                                float posterior_alpha, int32_t tie_break, float* logits, float* node_p,
                                float* node_H, int32_t* accept_len, int32_t* best_path, int32_t* best_node,
                                int32_t* accepted_tokens, int32_t* next_root, int32_t* dev_status,
                                const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                int32_t* kv_len, int32_t Hkv, int32_t D, int32_t Lmax, void* ws,
                                size_t ws_bytes, medusa_stream_t stream);

/* ------------------------------------------------------------------------
 * medusa_sample_next
 * The next token drawn from the top-p nucleus of the accepted node's
 * distribution softmax(z[best_node] / temperature), instead of its greedy
 * token (cnnetsun "Posterior probability evaluation": evaluate_posterior takes
 * top_p and a sampling mode; the pages define neither, so this library's
 * reading is stated here).  The nucleus is the shortest run of tokens in
 * descending probability (equal logits by the lower id) whose mass reaches
 * top_p; the draw picks by inverse CDF over the nucleus renormalised, tokens in
 * ascending id order: the first token whose running mass exceeds
 * uniform[b] times the nucleus mass.  The random draw is an input, so a step is
 * reproducible from its inputs; temperature 0 gives the greedy token.
 *   logits [B,T,V] fp32: medusa_verify_accept's logits output (the call must
 *   have been given a logits buffer); best_node [B] from the same call;
 *   uniform [B] fp32 in [0, 1) device; next_token [B] int32 out.
 *   0 < top_p <= 1.
 * ---------------------------------------------------------------------- */
int medusa_sample_next(const medusa_tree* tree, const float* logits, const int32_t* best_node,
                       const float* uniform, int32_t B, int32_t V, float temperature, float top_p,
                       int32_t* next_token, medusa_stream_t stream);

/* ------------------------------------------------------------------------
 * medusa_kv_commit
 * The kept branch continues the sequence (Ultralytics "Tree attention and
 * accepting tokens"; wiblog "Inference flow"): the K/V rows of the nodes
 * root..best_node[b] (depth 0..a) are copied to cache positions
 * kv_len[b]..kv_len[b]+a and kv_len[b] grows by a+1.  If that would pass
 * Lmax the request is left untouched and MEDUSA_DEV_KV_OVERFLOW is set.
 *   k_new, v_new [B,T,Hkv,D]; k_cache, v_cache [B,Hkv,Lmax,D] (in/out);
 *   kv_len [B] (in/out); best_node [B] from medusa_verify_accept.
 * ---------------------------------------------------------------------- */
int medusa_kv_commit(const medusa_tree* tree, const void* k_new, const void* v_new,
                     void* k_cache, void* v_cache, int32_t* kv_len, const int32_t* best_node,
                     int32_t B, int32_t Hkv, int32_t D, int32_t Lmax, medusa_dtype dtype,
                     int32_t* dev_status, medusa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MEDUSA_H_ */
