/*
 * ddt_oracle.h -- plain, slow fp64 CPU oracle of one DDTree verification round.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library.  It shares no code, header, table or
 * helper with the CUDA library in tree_speculative_decoding_02_gb300/csrc, and it
 * never includes or links that library.
 *
 * Sources (the method is described on these web pages; no code is printed there):
 *   [NOTES]  "DDTree on vLLM: candid research notes on tree speculation for Qwen3.6",
 *            sections "Why a tree instead of a chain", "Why hybrid attention makes it
 *            hard", "What broke along the way", "Where the next step is".
 *   [ARCH]   "From Tree-Based Speculative Decoding to Drafter Training: A Research
 *            Pivot in the DDTree Investigation", section "The Architecture of DDTree:
 *            Tree Construction and Verification".
 *   [CHALL]  "The Architecture of Speculation: Bridging DFlash and DDTree for
 *            Production Inference", section "The DDTree Integration Challenge".
 *   [VALID]  "The Moment of Truth: Validating DDTree Speculative Decoding on
 *            Qwen3.6-27B", section "The Path to This Message" (the serving stack's
 *            sampler is a linear-chain rejection sampler; a tree walk needs its own).
 *   [SPEC]   The pages name tree-walk rejection sampling but give no algorithm.  The
 *            acceptance rule used is speculative sampling's (Leviathan, Kalman and
 *            Matias, ICML 2023; Chen et al., 2023), applied over a node's children
 *            with point-mass drafts as in SpecInfer (Miao et al., ASPLOS 2024).
 *   [GDN]    The pages name Gated DeltaNet layers but print no formula.  The gated
 *            delta rule used here is the one of Yang, Kautz and Hatamizadeh, "Gated
 *            Delta Networks: Improving Mamba2 with Delta Rule" (ICLR 2025), in the
 *            form with L2-normalised q/k and a short causal convolution in front.
 *
 * All floating-point inputs are fp64 arrays (the Python side converts bf16/fp32
 * exactly).  All arithmetic is fp64.  Layouts are C row-major, outermost first.
 * Every function returns 0 on success or a DDTO_ERR_* code.
 *
 * Parity status: every function here is pinned by the CPU tests in
 * tests/test_oracle_pins.py (brute force, closed forms, invariants).
 */
#ifndef DDT_ORACLE_H
#define DDT_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DDTO_OK 0
#define DDTO_ERR_ARG 1
#define DDTO_ERR_TREE 7
#define DDTO_ERR_CAPACITY 3
#define DDTO_ERR_NONFINITE 6

/*
 * Best-first tree build ([ARCH]; [CHALL] item 2).
 *   logits      [B][D][V]  drafter logits of depths 1..D
 *   root_token  [B], prefix_len [B]
 * Outputs, N = budget + 1 rows per request (row 0 = root), W = ceil(N/32):
 *   token, parent, depth, position, rank [B][N]  (padding rows: -1)
 *   n_nodes [B]    rows in use (root included)
 *   anc [B][N][W]  bit j of row i set iff j is i or an ancestor of i
 *   score [B][N]   fp64 log-probability of the node's path (root 0, padding -inf)
 *   lse [B][D]     per-depth log-sum-exp
 *   margin [B]     score(last selected) - score(best unselected); +inf if none left
 *   margin_depth [B][2]  depths of those two nodes (-1 if absent)
 */
int ddto_build_tree(int B, int D, int V, int k, int budget,
                    const double* logits, const int32_t* root_token, const int32_t* prefix_len,
                    int32_t* token, int32_t* parent, int32_t* depth, int32_t* position,
                    int32_t* rank, int32_t* n_nodes, uint32_t* anc, double* score,
                    double* lse, double* margin, int32_t* margin_depth);

/*
 * Tree attention of one query row ([NOTES] "Why hybrid attention makes it hard";
 * [ARCH]): softmax(scale * q.K^T) V over the keys {prefix 0..P-1} and the tree rows j
 * whose bit is set in anc_row (j < n_nodes).
 *   q [d]; k_prefix, v_prefix [P][d] (row stride ld_prefix elements);
 *   k_tree, v_tree [n_nodes][d] (row stride ld_tree elements); out [d].
 */
int ddto_attn_row(int P, int n_nodes, int d, const double* q,
                  const double* k_prefix, const double* v_prefix, long ld_prefix,
                  const double* k_tree, const double* v_tree, long ld_tree,
                  const uint32_t* anc_row, double scale, double* out);

/*
 * Whole-batch tree attention, looping ddto_attn_row over every layer, request,
 * row < n_nodes and query head; rows >= n_nodes are written as zeros.
 *   q [L][B][N][Hq][d]; k_tree, v_tree [L][B][N][Hkv][d];
 *   k_cache, v_cache [L][B][Hkv][Pcap][d]; anc [B][N][W]; o [L][B][N][Hq][d].
 * Query head h reads kv head h / (Hq / Hkv).
 */
int ddto_tree_attn(int L, int B, int N, int Hq, int Hkv, int d, int Pcap,
                   const double* q, const double* k_tree, const double* v_tree,
                   const double* k_cache, const double* v_cache,
                   const int32_t* prefix_len, const int32_t* n_nodes, const uint32_t* anc,
                   double scale, double* o);

/*
 * Branch-local gated delta rule of one (layer, request, value head) unit
 * ([NOTES] "Why hybrid attention makes it hard", "Where the next step is"; [GDN]).
 * Each node runs the short conv over its own ancestor path and the gated delta rule
 * from its parent's state; the root starts from the committed state S0.
 *   x [N][C] pre-conv channels, C = 2*Hk*dk + Hv*dv, order q | k | v
 *   conv_w [C][K], conv_state [K-1][C] (oldest first)
 *   beta, decay [N][Hv]; S0 [dk][dv]; parent [N] (parent[0] = -1, parent[i] < i)
 *   o [N][dv] (rows >= n_nodes zero); S_node [N][dk][dv] or NULL.
 * Value head h reads key head h / (Hv / Hk).
 */
int ddto_gdn_unit(int N, int n_nodes, int Hk, int Hv, int dk, int dv, int K, int h,
                  const double* x, const double* conv_w, const double* conv_state,
                  const double* beta, const double* decay, const double* S0,
                  const int32_t* parent, double* o, double* S_node);

/*
 * Whole-batch tree GDN, looping ddto_gdn_unit over layers, requests and value heads.
 *   x [L][B][N][C]; conv_w [L][C][K]; conv_state [L][B][K-1][C];
 *   beta, decay [L][B][N][Hv]; S [L][B][Hv][dk][dv]; parent [B][N]; n_nodes [B];
 *   o [L][B][N][Hv][dv]; S_node [L][B][N][Hv][dk][dv] or NULL.
 */
int ddto_tree_gdn(int L, int B, int N, int Hk, int Hv, int dk, int dv, int K,
                  const double* x, const double* conv_w, const double* conv_state,
                  const double* beta, const double* decay, const double* S,
                  const int32_t* parent, const int32_t* n_nodes,
                  double* o, double* S_node);

/*
 * Greedy tree walk ([ARCH] "follow_verified_tree"; [NOTES] "What broke along the
 * way" for accepted vs emitted tokens).
 *   target_logits [B][N][V] or NULL; target_argmax_in [B][N] used when logits NULL.
 *   target_argmax_out [B][N] (may be NULL); acc_nodes [B][D+1] (root first, -1 pad);
 *   acc_len [B]; bonus [B]; emitted [B][D+1] (-1 pad); n_emitted [B].
 */
int ddto_walk(int B, int N, int V, int D, const double* target_logits,
              const int32_t* target_argmax_in, const int32_t* token, const int32_t* parent,
              const int32_t* n_nodes, int32_t* target_argmax_out, int32_t* acc_nodes,
              int32_t* acc_len, int32_t* bonus, int32_t* emitted, int32_t* n_emitted);
/* Flat-commit safe mode: as ddto_walk, but only a node's first (rank-0) child is ever
 * taken, so the accepted path is the agreeing prefix of the tree's flat chain. */
int ddto_walk_flat(int B, int N, int V, int D, const double* target_logits,
                   const int32_t* target_argmax_in, const int32_t* token, const int32_t* parent,
                   const int32_t* n_nodes, int32_t* target_argmax_out, int32_t* acc_nodes,
                   int32_t* acc_len, int32_t* bonus, int32_t* emitted, int32_t* n_emitted);

/*
 * Tree-walk rejection sampling ([VALID]; [SPEC]; [NOTES] "What broke along the way" for
 * accepted vs emitted tokens).  READING: at the visited node u (step s = depth of u),
 * p_u = softmax(target_logits[u] / T).  u's children are tried in row order; with R the
 * p_u-mass of the children already rejected, child i (token x_i, i counted from 0) is
 * accepted iff U[s][i] < p_u(x_i) / (1 - R), else R += p_u(x_i).  An accepted child is
 * the next node.  When every child is rejected (or u has none, or the walk has already
 * taken max-depth steps) the bonus token is the smallest id t, rejected children
 * skipped, whose running sum of p_u in id order exceeds U[s][C] * (1 - R); if rounding
 * leaves no such t, the largest id with positive residual mass.
 *   target_logits [B][N][V]; uniforms [B][D+1][C+1] in [0, 1); temperature T > 0.
 *   Outputs as ddto_walk, plus status [B] (DDTO_OK; DDTO_ERR_TREE for a node with more
 *   than C children, a repeated sibling token or a token outside [0, V);
 *   DDTO_ERR_NONFINITE for a non-finite logit in a row of the tree; the walk outputs
 *   are then the empty walk: acc_len 0, bonus -1, n_emitted 0) and margin [B]: the
 *   smallest distance, in probability, between a uniform's target and the threshold it
 *   was compared with over the request's decisions (for the bonus: to either end of the
 *   chosen token's interval of the running sum; 0 for the rounding fallback).
 */
int ddto_walk_sample(int B, int N, int V, int D, int C, double T, const double* target_logits,
                     const double* uniforms, const int32_t* token, const int32_t* parent,
                     const int32_t* n_nodes, int32_t* acc_nodes, int32_t* acc_len, int32_t* bonus,
                     int32_t* emitted, int32_t* n_emitted, double* margin, int32_t* status);

/*
 * Commit of the accepted path ([NOTES] "Why hybrid attention makes it hard",
 * "Where the next step is"; [ARCH] KV compaction).  In place:
 *   k_cache, v_cache [La][B][Hkv][Pcap][d]  rows prefix_len[b] + j <- tree row acc_nodes[b][j]
 *   S [Lg][B][Hv][dk][dv]  <- state after the last accepted node (sequential recurrence)
 *   conv_state [Lg][B][K-1][C] <- last K-1 raw inputs of [conv_state, path x]
 *   prefix_len [B] += acc_len + 1
 * src_row, dst_pos [B][A] (A = max accepted rows incl. root, -1 pad); status [B].
 * Requests with prefix_len + acc_len + 1 > Pcap get status DDTO_ERR_CAPACITY and are
 * left untouched.
 */
int ddto_commit(int La, int B, int N, int Hkv, int d, int Pcap,
                const double* k_tree, const double* v_tree, double* k_cache, double* v_cache,
                int Lg, int Hk, int Hv, int dk, int dv, int K,
                const double* x, const double* conv_w, const double* beta, const double* decay,
                double* S, double* conv_state,
                const int32_t* acc_nodes, const int32_t* acc_len, int A,
                int32_t* prefix_len, int32_t* src_row, int32_t* dst_pos, int32_t* status);

/* Paged KV caches ([NOTES] "Where the next step is": attention over paged KV blocks).
 * READING: the pages print no layout; a paged cache here is [L][num_pages][Hkv][page][d]
 * and row p of request b's prefix is row p % page of physical page
 * block_table[b][p / page].  ddto_gather_pages writes the contiguous cache
 * [L][B][Hkv][Pcap][d] that ddto_tree_attn / ddto_commit take (rows >= prefix_len[b]
 * zero); ddto_scatter_pages writes rows [0, n_rows[b]) of a contiguous cache back into
 * the pages.  Both return DDTO_ERR_ARG for a block-table entry outside [0, num_pages)
 * or a row past the capacity. */
int ddto_gather_pages(int L, int B, int Hkv, int d, int page, int num_pages, int max_pages,
                      const double* pages, const int32_t* block_table, const int32_t* prefix_len,
                      int Pcap, double* cache);
int ddto_scatter_pages(int L, int B, int Hkv, int d, int page, int num_pages, int max_pages,
                       const double* cache, int Pcap, const int32_t* block_table,
                       const int32_t* n_rows, double* pages);

/* Rotary embedding of tree rows by depth ([NOTES] "Where the next step is": position and
 * RoPE correctness by branch depth).  READING: the half-split convention of Qwen-style
 * models.  In place on x [L][B][N][H][d]: for node n < n_nodes[b], i < rot/2,
 * a = position[b][n] * theta^(-2i/rot): (x[i], x[i+rot/2]) <- (x[i] cos a - x[i+rot/2] sin a,
 * x[i+rot/2] cos a + x[i] sin a); other channels and padding rows unchanged. */
int ddto_rope_tree(int L, int B, int N, int H, int d, int rot, double theta,
                   const int32_t* position, const int32_t* n_nodes, double* x);

#ifdef __cplusplus
}
#endif
#endif
