/*
 * ddt.h -- C ABI of the GB300 (sm_103a) DDTree verification-round library.
 *
 * One verification round of DDTree tree-speculative decoding for a hybrid target
 * made of full-attention and Gated DeltaNet (GDN) layers, as five stream-ordered
 * calls:
 *
 *   ddt_build_tree   best-first draft tree from the drafter's per-depth logits
 *   ddt_tree_attn    tree attention: prefix KV + own ancestors, never siblings
 *   ddt_tree_gdn     branch-local gated delta rule + short conv, scratch-only state
 *   ddt_walk_accept  greedy tree walk against the target's argmax
 *                    (ddt_walk_accept_sample: the same walk at a temperature, by
 *                    rejection sampling over each node's children)
 *   ddt_commit       copy only the accepted path's KV / recurrent state
 *
 * Sources (web pages; no code is printed on them):
 *   [NOTES] "DDTree on vLLM: candid research notes on tree speculation for Qwen3.6"
 *           -- "Why a tree instead of a chain", "Why hybrid attention makes it hard",
 *           "What broke along the way", "Where the next step is".
 *   [ARCH]  "From Tree-Based Speculative Decoding to Drafter Training: A Research Pivot
 *           in the DDTree Investigation" -- "The Architecture of DDTree: Tree
 *           Construction and Verification".
 *   [CHALL] "The Architecture of Speculation: Bridging DFlash and DDTree for Production
 *           Inference" -- "The DDTree Integration Challenge".
 *   [GDN]   Yang, Kautz, Hatamizadeh, "Gated Delta Networks" (ICLR 2025): the gated
 *           delta rule, which the pages name but do not print.
 *
 * Conventions for every call:
 *   - All array pointers are DEVICE pointers, contiguous, C row-major with the
 *     shapes given below (outermost first).  The caller owns and allocates every
 *     buffer, including workspaces; the library allocates no device memory and keeps
 *     no global state (ddt_build_tree_noalloc's fixed scratch array aside).  Calls are
 *     thread-safe.
 *   - Work is enqueued on `stream`; nothing synchronises the host.  Results and the
 *     per-request `status` words are valid once the stream has reached the call.
 *   - Argument errors found on the host (null pointers, unsupported sizes, short
 *     workspace) return an error before anything is launched.  Data errors found on
 *     the device (non-finite logits, malformed trees, cache overflow) are written to
 *     `status[b]` as a ddt_status code, per request; kernels never trap.
 *   - N = budget + 1 tree rows per request.  Row 0 is the root (the last emitted
 *     token, not yet in the cache); rows 1..n_nodes[b]-1 are drafted nodes numbered
 *     breadth first (depth, then parent row, then rank), so every parent row is
 *     smaller than its children's.  Rows >= n_nodes[b] are padding.
 *   - W = ceil(N / 32) mask words per row.
 */
#ifndef DDT_H
#define DDT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ddt_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
    DDT_OK = 0,
    DDT_ERR_INVALID_ARG = 1, /* null pointer, bad size, short workspace */
    DDT_ERR_UNSUPPORTED = 2, /* size/dtype combination not compiled in */
    DDT_ERR_CAPACITY = 3,    /* prefix_len + committed rows would exceed the cache */
    DDT_ERR_CUDA = 4,        /* a launch failed; see cudaGetLastError semantics */
    DDT_ERR_TIMEOUT = 5,     /* a bounded device wait gave up (per request, tensor-core kernels) */
    DDT_ERR_NONFINITE = 6,   /* NaN or +-Inf logits */
    DDT_ERR_TREE = 7         /* malformed tree arrays (parent >= child, bad token) */
} ddt_status;

typedef enum { DDT_F32 = 0, DDT_BF16 = 1 } ddt_dtype;

/* Text of a status code (static storage). */
const char* ddt_status_string(ddt_status s);

/* Library version, e.g. "ddt 0.1 sm_103a". */
const char* ddt_version(void);

/* Number of kernel launches the library has issued in this process so far, over all
 * threads, streams and devices (launches that CUDA rejected included).  A caller takes
 * the difference around a region to count the kernels that region launched.  No
 * counterpart in the pages: bookkeeping for measurement. */
uint64_t ddt_launch_count(void);

/* Runs one bounded device wait on an mbarrier that nothing ever signals -- the same
 * wait, with the same limit (about one second of SM clock cycles), that every pipeline
 * barrier of the tensor-core kernels uses -- and writes its outcome to status[0]:
 * DDT_ERR_TIMEOUT when the wait gave up, as it must.  The kernel then returns normally,
 * so the context stays usable.  This exercises the failure path of the bounded waits
 * without a fault.  status: one int32 on the device.  Returns DDT_ERR_INVALID_ARG for a
 * null status, DDT_ERR_CUDA if the launch fails.  No counterpart in the pages. */
ddt_status ddt_wait_selftest(int32_t* status, ddt_stream_t stream);

/* ---------------------------------------------------------------------------------
 * ddt_build_tree -- [ARCH] best-first tree construction and flattening; [CHALL] 2.
 *
 * For each depth d = 1..D of each request: LSE_d = log sum_v exp(logit_d[v]); the
 * depth's top_k tokens by (logit desc, token id asc).  A node is a path (t_1..t_n)
 * with t_i among depth i's top_k; its score is log prod_i p_i(t_i) =
 * sum_i logit_i(t_i) - sum_i LSE_i, each sum formed in fp64 depth 1 first.  The
 * `budget` nodes taken are those a best-first max-heap pops, seeded with the best
 * depth-1 token and pushing, per pop, the next-ranked sibling and the best child;
 * exact score ties go to the lexicographically smaller token path.  If the lattice
 * holds fewer than `budget` nodes, all of it is taken.
 *
 *   draft_logits [B][D][V] (dtype)       root_token [B], prefix_len [B] int32
 * Outputs (int32 unless noted), padding rows = -1:
 *   token [B][N], parent [B][N] (root -1), depth [B][N] (root 0),
 *   position [B][N] = prefix_len[b] + depth, n_nodes [B] (root included),
 *   anc [B][N][W] uint32: bit j of row i set iff row j is row i or an ancestor of it,
 *   score [B][N] double (root 0, padding -inf) -- may be NULL,
 *   status [B]: DDT_OK or DDT_ERR_NONFINITE (then the tree is the root alone).
 * Limits: 1 <= D <= 64, 1 <= top_k <= min(32, V), 0 <= budget <= 1023.
 * workspace: ddt_build_tree_workspace(B, D, V, top_k) bytes, 16-byte aligned.
 * ------------------------------------------------------------------------------- */
size_t ddt_build_tree_workspace(int B, int D, int V, int top_k);
ddt_status ddt_build_tree(int B, int D, int V, int top_k, int budget, ddt_dtype dtype,
                          const void* draft_logits, const int32_t* root_token,
                          const int32_t* prefix_len, int32_t* token, int32_t* parent,
                          int32_t* depth, int32_t* position, int32_t* n_nodes, uint32_t* anc,
                          double* score, int32_t* status, void* workspace, size_t ws_bytes,
                          ddt_stream_t stream);

/* ---------------------------------------------------------------------------------
 * ddt_build_tree_noalloc -- not part of the method (the pages have no counterpart): the
 * ddt_build_tree above for callers that cannot allocate device memory, such as a plain
 * C host without a device allocator, or a plugin inside a process whose GPU memory is
 * owned by another runtime, or a decode loop that must not call cudaMalloc/cudaFree
 * because they synchronise the device.  Same arguments and results as ddt_build_tree,
 * without the workspace: the scratch is a fixed 4 MiB device array inside the library,
 * present on every GPU that loads the library until the process exits.
 *   - The first call on a device looks up that array's device address (with the device
 *     current) and caches it with the CUDA context it belongs to; a call made in another
 *     context of that device (after cudaDeviceReset, or once the primary context was
 *     released and created again) looks it up anew.  Make the first call in a context
 *     before any stream capture.
 *   - Every call on a device shares the array, which keeps the last call's contents:
 *     calls whose kernels overlap on the GPU race on it and must be ordered by the caller.
 *   - Returns DDT_ERR_CAPACITY, before launching anything, when the call needs more
 *     than 4 MiB (ddt_build_tree_workspace(B, D, V, top_k) = B*D*(16 + 8*top_k) bytes,
 *     rounded up to 256, > 4 MiB), e.g. B = 32, D = 15 needs 38 KiB with top_k = 8;
 *     B = 2048, D = 64, top_k = 32 (35 MiB) is refused.
 *   - Allocates nothing (no cudaMalloc, no allocating library call).
 * ------------------------------------------------------------------------------- */
ddt_status ddt_build_tree_noalloc(int B, int D, int V, int top_k, int budget, ddt_dtype dtype,
                                  const void* draft_logits, const int32_t* root_token,
                                  const int32_t* prefix_len, int32_t* token, int32_t* parent,
                                  int32_t* depth, int32_t* position, int32_t* n_nodes,
                                  uint32_t* anc, double* score, int32_t* status,
                                  ddt_stream_t stream);

/* ---------------------------------------------------------------------------------
 * ddt_tree_attn -- [NOTES] "Why hybrid attention makes it hard": each tree row attends
 * to the committed prefix plus its own ancestors (and itself), never its siblings;
 * [ARCH] the ancestor-only attention mask of the flattened tree.
 *
 * For layer l, request b, row i < n_nodes[b], query head h (kv head g = h / (Hq/Hkv)):
 *   o = softmax(scale * q . K^T) V over keys {k_cache rows 0..prefix_len[b]-1} and
 *       {k_tree rows j : bit j of anc[b][i]}.
 * scale is the caller's softmax scale (1/sqrt(d) for standard attention); the library
 * applies it as given and supplies no default.  Inputs are taken after any rotary
 * embedding.
 *   q [L][B][N][Hq][d], k_tree, v_tree [L][B][N][Hkv][d]  (in_dtype)
 *   k_cache, v_cache [L][B][Hkv][Pcap][d] (in_dtype): only rows < prefix_len[b] are
 *     read; the rest may hold anything.  Tree rows >= n_nodes[b] are never read.
 *   prefix_len, n_nodes [B]; anc [B][N][W] as written by ddt_build_tree.
 *   o [L][B][N][Hq][d] (out_dtype); padding rows are written as zeros.
 *   status [B]: DDT_ERR_CAPACITY if prefix_len[b] is outside [0, Pcap], DDT_ERR_TREE
 *     if n_nodes[b] is outside [1, N] (the request's output rows are then zero).
 * d in {64, 128, 256}; Hq % Hkv == 0; N <= 1024.
 * workspace: ddt_tree_attn_workspace(...) bytes (split-KV partials), 16-byte aligned.
 * ------------------------------------------------------------------------------- */
size_t ddt_tree_attn_workspace(int n_layers, int B, int N, int Hq, int Hkv, int d, int Pcap);
ddt_status ddt_tree_attn(int n_layers, int B, int N, int Hq, int Hkv, int d, int Pcap,
                         ddt_dtype in_dtype, ddt_dtype out_dtype, const void* q,
                         const void* k_tree, const void* v_tree, const void* k_cache,
                         const void* v_cache, const int32_t* prefix_len, const int32_t* n_nodes,
                         const uint32_t* anc, float scale, void* o, int32_t* status,
                         void* workspace, size_t ws_bytes, ddt_stream_t stream);

/* ---------------------------------------------------------------------------------
 * ddt_tree_attn_paged -- ddt_tree_attn over a paged prefix cache ([NOTES] "Where the
 * next step is": fused ancestor-mask branch attention over paged KV blocks).
 *
 * Same result as ddt_tree_attn where request b's prefix row p (p < prefix_len[b]) is
 *   k_pages[l][block_table[b][p / page_size]][g][p % page_size][:]   (same for v).
 *   k_pages, v_pages [L][num_pages][Hkv][page_size][d] (bf16; head-major pages).
 *   block_table [B][max_pages] int32: physical page of each logical page; only the
 *     first ceil(prefix_len[b] / page_size) entries are read.  Rows of the last page past
 *     prefix_len[b] may hold anything (they are masked, and their V rows are zeroed
 *     before use, so NaN there does no harm).
 *   page_size: 8, 16, 32, or a multiple of 64.  Capacity is max_pages * page_size.
 *   status [B]: as ddt_tree_attn, plus DDT_ERR_INVALID_ARG when a block-table entry
 *     the prefix needs is outside [0, num_pages) (that request's rows are then zero).
 * bf16 inputs, d in {64, 128, 256} only (DDT_ERR_UNSUPPORTED otherwise).
 * workspace: ddt_tree_attn_paged_workspace(...) bytes, 16-byte aligned.
 * ------------------------------------------------------------------------------- */
size_t ddt_tree_attn_paged_workspace(int n_layers, int B, int N, int Hq, int Hkv, int d,
                                     int page_size, int max_pages);
ddt_status ddt_tree_attn_paged(int n_layers, int B, int N, int Hq, int Hkv, int d,
                               int page_size, int num_pages, int max_pages,
                               ddt_dtype in_dtype, ddt_dtype out_dtype, const void* q,
                               const void* k_tree, const void* v_tree, const void* k_pages,
                               const void* v_pages, const int32_t* block_table,
                               const int32_t* prefix_len, const int32_t* n_nodes,
                               const uint32_t* anc, float scale, void* o, int32_t* status,
                               void* workspace, size_t ws_bytes, ddt_stream_t stream);

/* ---------------------------------------------------------------------------------
 * ddt_tree_attn_rope / ddt_tree_attn_paged_rope -- [NOTES] "Where the next step is":
 * branch attention over (paged) KV with rotary embedding by branch depth, fused.
 *
 * Same results as ddt_rope_tree on q followed by ddt_tree_attn (resp. _paged) -- bit for
 * bit: q is given BEFORE rotary embedding and each of its rows is rotated at its node's
 * position (position [B][N], as written by ddt_build_tree) while the kernel stages it, in
 * the arithmetic of ddt_rope_tree, then rounded to bf16 once.  q is never committed, so
 * nothing else changes; k_tree must already be rotated (ddt_rope_tree with q = NULL
 * rotates the keys alone, in place, which the commit then copies).
 *   rot_dim: a multiple of 16, 16 <= rot_dim <= d; theta > 1 (ddt_rope_tree's meaning).
 *   bf16 with d in {128, 256} only (DDT_ERR_UNSUPPORTED otherwise).
 *   workspace: the workspace of the plain call rounded up to 256 bytes, plus
 *     B * N * rot_dim * 4 bytes for the per-row cos/sin table; 16-byte aligned.
 * All other arguments, outputs and statuses are those of ddt_tree_attn / _paged.
 * ------------------------------------------------------------------------------- */
ddt_status ddt_tree_attn_rope(int n_layers, int B, int N, int Hq, int Hkv, int d, int Pcap,
                              ddt_dtype in_dtype, ddt_dtype out_dtype, const void* q,
                              const void* k_tree, const void* v_tree, const void* k_cache,
                              const void* v_cache, const int32_t* prefix_len,
                              const int32_t* n_nodes, const uint32_t* anc, const int32_t* position,
                              int rot_dim, double theta, float scale, void* o, int32_t* status,
                              void* workspace, size_t ws_bytes, ddt_stream_t stream);
ddt_status ddt_tree_attn_paged_rope(int n_layers, int B, int N, int Hq, int Hkv, int d,
                                    int page_size, int num_pages, int max_pages,
                                    ddt_dtype in_dtype, ddt_dtype out_dtype, const void* q,
                                    const void* k_tree, const void* v_tree, const void* k_pages,
                                    const void* v_pages, const int32_t* block_table,
                                    const int32_t* prefix_len, const int32_t* n_nodes,
                                    const uint32_t* anc, const int32_t* position, int rot_dim,
                                    double theta, float scale, void* o, int32_t* status,
                                    void* workspace, size_t ws_bytes, ddt_stream_t stream);

/* ---------------------------------------------------------------------------------
 * ddt_rope_tree -- [NOTES] "Where the next step is": position and RoPE correctness by
 * branch depth.  Rotary embedding of the tree rows, in place, at each node's own position
 * (position[b][n] from ddt_build_tree: prefix_len + depth, shared by siblings).
 *
 * For every layer, request b, node n < n_nodes[b], and every head row x of q
 * [L][B][N][Hq][d] and of k_tree [L][B][N][Hkv][d] (dtype):
 *   for i < rot_dim/2, with a = position[b][n] * theta^(-2i/rot_dim):
 *     x[i] <- x[i] cos a - x[i + rot_dim/2] sin a,
 *     x[i + rot_dim/2] <- x[i + rot_dim/2] cos a + x[i] sin a;   channels >= rot_dim kept.
 * READING: the pages give no rotary formula; this is the half-split convention of
 * Qwen-style models, with partial rotation (rot_dim < d) allowed.  Rows of padding
 * nodes are left unchanged.  Call it before ddt_tree_attn / ddt_commit so that the
 * committed keys are the rotated ones.  q may be NULL: then only the keys are rotated
 * (for the fused ddt_tree_attn_rope, which rotates q itself).  rot_dim even,
 * 2 <= rot_dim <= d; theta > 1.
 * ------------------------------------------------------------------------------- */
ddt_status ddt_rope_tree(int n_layers, int B, int N, int Hq, int Hkv, int d, int rot_dim,
                         double theta, ddt_dtype dtype, const int32_t* position,
                         const int32_t* n_nodes, void* q, void* k_tree, ddt_stream_t stream);

/* ---------------------------------------------------------------------------------
 * ddt_tree_gdn -- [NOTES] "Why hybrid attention makes it hard" / "Where the next step
 * is": each node reads the GDN and conv state of its parent and writes scratch, never
 * the committed state; [GDN] the gated delta rule.
 *
 * Per layer l, request b, value head h (key head g = h / (Hv/Hk)), node n (parent p):
 *   conv: y[c] = SiLU(sum_j conv_w[c][j] * in_j[c]), j = 0..K-1, in_{K-1} = x_n,
 *         in_{K-2} = x_p, ... along the node's ancestor path; taps past the root read
 *         conv_state (row K-2 = newest).
 *   q^ = y_q / sqrt(|y_q|^2 + 1e-6) / sqrt(dk),  k^ = y_k / sqrt(|y_k|^2 + 1e-6),  v = y_v
 *   S_n = decay_n * S_p + (beta_n * (v - decay_n * S_p k^)) k^T     (S_root's parent = S)
 *   o_n = S_n q^
 * State matrices are stored value-major: S[j][i], j < dv value channel, i < dk key
 * channel, so o = S q and the update is a rank-one term u k^T.
 *   x [L][B][N][C] (in_dtype), C = 2*Hk*dk + Hv*dv, channel order q | k | v
 *   conv_w [L][C][K] (in_dtype), conv_state [L][B][K-1][C] (in_dtype, oldest first)
 *   beta, decay [L][B][N][Hv] fp32;  S [L][B][Hv][dv][dk] fp32 (read only)
 *   parent [B][N], n_nodes [B] as written by ddt_build_tree
 *   o [L][B][N][Hv][dv] (out_dtype); padding rows are zeros.
 *   S_node_debug: NULL, or [L][B][N][Hv][dv][dk] fp32 that receives every node's own
 *     branch-local state S_n, computed the literal way: node n reads its parent's state
 *     from this buffer (the root reads S) and writes its own row, parents before
 *     children.  A debugging aid for small trees (it writes N states per head, so it is
 *     not for full-size workloads); the fast path never forms these states.  Padding
 *     rows are zeros.  The o outputs are those of the normal path either way.
 *   status [B]: DDT_ERR_TREE for a malformed parent array, DDT_ERR_UNSUPPORTED for a
 *     tree deeper than the head-128 limit below (that request's outputs are then zero).
 * Limits: dk, dv in {32, 64, 128} (dk = dv = 128 runs on the tensor cores and takes
 * trees of depth <= 16, i.e. drafter depth <= 16; other sizes take depth <= 32);
 * 1 <= K <= 8; N <= 128.
 * ------------------------------------------------------------------------------- */
size_t ddt_tree_gdn_workspace(int n_layers, int B, int N, int Hk, int Hv, int dk, int dv);
ddt_status ddt_tree_gdn(int n_layers, int B, int N, int Hk, int Hv, int dk, int dv, int conv_k,
                        ddt_dtype in_dtype, ddt_dtype out_dtype, const void* x,
                        const void* conv_w, const void* conv_state, const float* beta,
                        const float* decay, const float* S, const int32_t* parent,
                        const int32_t* n_nodes, void* o, float* S_node_debug, int32_t* status,
                        void* workspace, size_t ws_bytes, ddt_stream_t stream);

/* ---------------------------------------------------------------------------------
 * ddt_walk_accept -- [ARCH] follow_verified_tree; [NOTES] "What broke along the way"
 * (accepted and emitted tokens are kept apart).
 *
 * t_i = argmax_v target_logits[b][i][v] (ties to the lower id).  Starting at the root,
 * move to the child whose token equals t_cur while one exists.  a = depth reached.
 *   target_logits [B][N][V] (dtype) or NULL; target_argmax [B][N]: written when
 *     target_logits is given, read otherwise.
 *   token, parent, n_nodes as written by ddt_build_tree.
 * Outputs: acc_nodes [B][A] (rows root, ..., last accepted; -1 pad), acc_len [B] = a,
 *   bonus [B] = t at the last accepted row (emitted, not an accepted draft),
 *   emitted [B][A] = tokens of accepted rows 1..a then bonus (-1 pad),
 *   n_emitted [B] = a + 1, status [B] (DDT_ERR_NONFINITE, DDT_ERR_TREE).
 * A = max_accept + 1 columns; max_accept >= the tree depth (D).
 * workspace: ddt_walk_accept_workspace(B, N, V) bytes.
 * ------------------------------------------------------------------------------- */
size_t ddt_walk_accept_workspace(int B, int N, int V);
ddt_status ddt_walk_accept(int B, int N, int V, int max_accept, ddt_dtype dtype,
                           const void* target_logits, int32_t* target_argmax,
                           const int32_t* token, const int32_t* parent, const int32_t* n_nodes,
                           int32_t* acc_nodes, int32_t* acc_len, int32_t* bonus,
                           int32_t* emitted, int32_t* n_emitted, int32_t* status,
                           void* workspace, size_t ws_bytes, ddt_stream_t stream);

/* ddt_walk_accept_flat -- the flat-commit safe mode ([NOTES] "What broke along the way":
 * full non-flat branch commit through the hybrid state is kept behind a research switch).
 * Same arguments and outputs as ddt_walk_accept, but the walk only ever descends into a
 * node's first child (its rank-0 child: children are numbered by rank), so the accepted
 * path is the longest agreeing prefix of the flat DFlash chain inside the tree, and a
 * round behaves exactly like flat DFlash verification of that chain. */
ddt_status ddt_walk_accept_flat(int B, int N, int V, int max_accept, ddt_dtype dtype,
                                const void* target_logits, int32_t* target_argmax,
                                const int32_t* token, const int32_t* parent,
                                const int32_t* n_nodes, int32_t* acc_nodes, int32_t* acc_len,
                                int32_t* bonus, int32_t* emitted, int32_t* n_emitted,
                                int32_t* status, void* workspace, size_t ws_bytes,
                                ddt_stream_t stream);

/* ---------------------------------------------------------------------------------
 * ddt_walk_accept_sample -- tree-walk rejection sampling at a temperature.
 * ["The Moment of Truth: Validating DDTree Speculative Decoding on Qwen3.6-27B",
 * "The Path to This Message": the serving stack samples with a linear-chain rejection
 * sampler; a tree needs a walk of its own.  The pages give no algorithm: the rule here
 * is speculative sampling's (Leviathan et al. and Chen et al., 2023) over each visited
 * node's children, whose draft is a point mass (SpecInfer, Miao et al., 2024).]
 *
 * At the visited node u (step s = depth of u, root first), p_u = softmax(logits[u] / T).
 * u's children are tried in row order (rank order for ddt_build_tree's trees); with R
 * the p_u-mass of the children already rejected, child i (counted from 0, token x_i) is
 * accepted iff U[b][s][i] < p_u(x_i) / (1 - R); a rejected child adds p_u(x_i) to R.  An
 * accepted child is the next node.  When every child is rejected (or u has none, or the
 * walk has taken max_accept steps), the bonus token is the smallest id, rejected
 * children skipped, whose running sum of p_u in id order exceeds U[b][s][C] * (1 - R).
 * Every emitted token is then distributed as the target's own p at its position.
 *   target_logits [B][N][V] (dtype); uniforms [B][A][C + 1] fp32 in [0, 1), C =
 *     max_children (the caller's random numbers: the same uniforms give the same walk).
 *   temperature T > 0 with 1/T finite in fp32 (else DDT_ERR_INVALID_ARG).
 *   token, parent, n_nodes as written by ddt_build_tree.
 * Outputs as ddt_walk_accept (acc_nodes, acc_len, bonus, emitted, n_emitted, status);
 * status [B]: DDT_ERR_TREE for a malformed tree, a node with more than C children, a
 * token repeated among one node's children or a token outside [0, V); DDT_ERR_NONFINITE
 * for a NaN or +-inf logit in any row of the tree; the walk is then empty (acc_len 0,
 * bonus -1, n_emitted 0).
 * Precision: each term exp((l - m) / T) is taken in fp32 as 2^((l - m) * s2), s2 =
 * log2(e) / T rounded to fp32, by the hardware base-2 exponential (relative error about
 * 2^-22); the per-row normaliser sums them in fp32 within each
 * 2048-entry unit and in fp64 across units; each comparison of a probability with a
 * uniform is in fp64.  A decision whose margin is below about 2e-6 may therefore differ
 * from an exact one.
 * Limits: 1 <= C <= 32, max_accept <= 64, N <= 1024, B <= 65535.
 * workspace: ddt_walk_accept_sample_workspace(B, N, V) bytes, 16-byte aligned.
 * ------------------------------------------------------------------------------- */
size_t ddt_walk_accept_sample_workspace(int B, int N, int V);
ddt_status ddt_walk_accept_sample(int B, int N, int V, int max_accept, int max_children,
                                  float temperature, ddt_dtype dtype, const void* target_logits,
                                  const float* uniforms, const int32_t* token,
                                  const int32_t* parent, const int32_t* n_nodes,
                                  int32_t* acc_nodes, int32_t* acc_len, int32_t* bonus,
                                  int32_t* emitted, int32_t* n_emitted, int32_t* status,
                                  void* workspace, size_t ws_bytes, ddt_stream_t stream);

/* ---------------------------------------------------------------------------------
 * ddt_commit -- [NOTES] "Why hybrid attention makes it hard": once a path is accepted,
 * only that path is copied into the contiguous KV and recurrent buffers; [ARCH] KV
 * compaction.  In place, per request b with a = acc_len[b], P = prefix_len[b]:
 *   KV: for every attention layer and kv head, cache row P + j <- tree row
 *       acc_nodes[b][j], j = 0..a (root first).  The bonus token is not committed.
 *   GDN: S[l][b][h] <- the state after the last accepted row, i.e. the rule of
 *       ddt_tree_gdn run along acc_nodes[b][0..a] from the committed state.
 *   conv_state[l][b] <- the last K-1 rows of [conv_state ; x rows of the path].
 *   prefix_len[b] <- P + a + 1;  src_row[b][j] = acc_nodes[b][j], dst_pos[b][j] = P + j
 *   (-1 pad).
 * If P + a + 1 > Pcap (with attention layers) the request is left untouched and
 * status[b] = DDT_ERR_CAPACITY.
 * Attention part: n_attn_layers (may be 0), Hkv, d, Pcap, kv_dtype, k_tree, v_tree
 *   [La][B][N][Hkv][d], k_cache, v_cache [La][B][Hkv][Pcap][d].
 * GDN part: n_gdn_layers (may be 0), Hk, Hv, dk, dv, conv_k, x_dtype, x [Lg][B][N][C],
 *   conv_w [Lg][C][K], beta, decay [Lg][B][N][Hv] fp32, S [Lg][B][Hv][dv][dk] fp32,
 *   conv_state [Lg][B][K-1][C].
 * acc_nodes [B][A], acc_len [B] as written by ddt_walk_accept.
 * ------------------------------------------------------------------------------- */
ddt_status ddt_commit(int B, int N, int A,
                      int n_attn_layers, int Hkv, int d, int Pcap, ddt_dtype kv_dtype,
                      const void* k_tree, const void* v_tree, void* k_cache, void* v_cache,
                      int n_gdn_layers, int Hk, int Hv, int dk, int dv, int conv_k,
                      ddt_dtype x_dtype, const void* x, const void* conv_w, const float* beta,
                      const float* decay, float* S, void* conv_state,
                      const int32_t* acc_nodes, const int32_t* acc_len, int32_t* prefix_len,
                      int32_t* src_row, int32_t* dst_pos, int32_t* status, ddt_stream_t stream);

/* ddt_commit_paged -- ddt_commit for paged KV caches (the layout of ddt_tree_attn_paged):
 * accepted row j of request b goes to position prefix_len[b] + j, i.e. row
 * (prefix_len[b] + j) % page_size of page block_table[b][(prefix_len[b] + j) / page_size]
 * of k_pages / v_pages [L][num_pages][Hkv][page_size][d].  Capacity is max_pages *
 * page_size; a block-table entry outside [0, num_pages) for a position being written
 * makes the request's status DDT_ERR_INVALID_ARG and nothing of it is committed.  The
 * GDN and conv-state part, the outputs and the other statuses are those of ddt_commit. */
ddt_status ddt_commit_paged(int B, int N, int A, int n_attn_layers, int Hkv, int d, int page_size,
                            int num_pages, int max_pages, const int32_t* block_table,
                            ddt_dtype kv_dtype, const void* k_tree, const void* v_tree,
                            void* k_pages, void* v_pages, int n_gdn_layers, int Hk, int Hv, int dk,
                            int dv, int conv_k, ddt_dtype x_dtype, const void* x, const void* conv_w,
                            const float* beta, const float* decay, float* S, void* conv_state,
                            const int32_t* acc_nodes, const int32_t* acc_len, int32_t* prefix_len,
                            int32_t* src_row, int32_t* dst_pos, int32_t* status, ddt_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DDT_H */
