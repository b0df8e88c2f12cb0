// kernels.h -- internal launchers of the DDTree round library (host side).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ddt.h"

namespace ddt {


constexpr int kMaxDepth = 64;      // deepest tree the build supports
constexpr int kMaxTopK = 32;
constexpr int kMaxBudget = 1023;
constexpr int kMaxRows = 1024;     // N = budget + 1
constexpr int kMaxAccept = kMaxDepth;  // accepted rows a commit takes (acc_len <= tree depth)
constexpr int kGdnMaxNodes = 128;
constexpr int kGdnMaxDepth = 32;

// Launch counter: every launch site passes its grid through counted(), so that
// ddt_launch_count() can report how many kernels this library has put on streams.
void note_launch();
template <typename G>
inline G counted(G grid) {
    note_launch();
    return grid;
}

size_t build_ws_bytes(int B, int D, int V, int k);
size_t build_tree_smem(int D, int k, int budget);
cudaError_t launch_build_tree(int B, int D, int V, int k, int budget, ddt_dtype dtype, const void* logits,
                              const int32_t* root_token, const int32_t* prefix_len, int32_t* token,
                              int32_t* parent, int32_t* depth, int32_t* position, int32_t* n_nodes,
                              uint32_t* anc, double* score, int32_t* status, void* ws, cudaStream_t st);

size_t walk_sample_ws_bytes(int B, int N, int V);
cudaError_t launch_walk_sample(int B, int N, int V, int A, int C, float temperature, ddt_dtype dtype,
                               const void* logits, const float* uniforms, const int32_t* token,
                               const int32_t* parent, const int32_t* n_nodes, int32_t* acc_nodes, int32_t* acc_len,
                               int32_t* bonus, int32_t* emitted, int32_t* n_emitted, int32_t* status, void* ws,
                               cudaStream_t st);
size_t walk_ws_bytes(int B, int N, int V);
cudaError_t launch_walk(int B, int N, int V, int A, ddt_dtype dtype, const void* logits, int32_t* targ,
                        const int32_t* token, const int32_t* parent, const int32_t* n_nodes, int32_t* acc_nodes,
                        int32_t* acc_len, int32_t* bonus, int32_t* emitted, int32_t* n_emitted, int32_t* status,
                        void* ws, int flat, cudaStream_t st);

cudaError_t launch_attn_simt(int L, int B, int N, int Hq, int Hkv, int d, int Pcap, ddt_dtype in, ddt_dtype out,
                             const void* q, const void* k_tree, const void* v_tree, const void* k_cache,
                             const void* v_cache, const int32_t* prefix_len, const int32_t* n_nodes,
                             const uint32_t* anc, float scale, void* o, int32_t* status, cudaStream_t st);

// paged prefix caches: positions p of request b live in page block_table[b][p / page_rows]
struct AttnPaging {
    int page_rows, num_pages, max_pages;
    const int32_t* block_table;  // [B][max_pages]
};
// rotary embedding of q applied by the attention kernel while it stages q
struct AttnRope {
    int rot;             // rotated channels (a multiple of 16, <= d)
    const float* table;  // [B][N][rot] from launch_rope_table
};
cudaError_t launch_attn_tc_paged(int L, int B, int N, int Hq, int Hkv, int d, const AttnPaging& pg, ddt_dtype out,
                                 const void* q, const void* k_tree, const void* v_tree, const void* k_pages,
                                 const void* v_pages, const int32_t* prefix_len, const int32_t* n_nodes,
                                 const uint32_t* anc, float scale, void* o, int32_t* status, void* ws,
                                 size_t ws_bytes, cudaStream_t st, const AttnRope* rope = nullptr);
size_t attn_tc_ws_bytes(int L, int B, int N, int Hq, int Hkv, int d, int Pcap);
bool attn_tc_supported(int d, ddt_dtype in);
cudaError_t launch_attn_tc(int L, int B, int N, int Hq, int Hkv, int d, int Pcap, ddt_dtype out, const void* q,
                           const void* k_tree, const void* v_tree, const void* k_cache, const void* v_cache,
                           const int32_t* prefix_len, const int32_t* n_nodes, const uint32_t* anc, float scale,
                           void* o, int32_t* status, void* ws, size_t ws_bytes, cudaStream_t st,
                           const AttnRope* rope = nullptr);

// one bounded wait on an mbarrier nothing signals; status[0] = its outcome
cudaError_t launch_wait_selftest(int32_t* status, cudaStream_t st);
cudaError_t launch_rope_tree(int L, int B, int N, int Hq, int Hkv, int d, int rot, double theta, ddt_dtype dtype,
                             const int32_t* position, const int32_t* n_nodes, void* q, void* k, cudaStream_t st);
cudaError_t launch_rope_table(int B, int N, int rot, double theta, const int32_t* position, const int32_t* n_nodes,
                              float* table, cudaStream_t st);
bool gdn_tc_supported(int N, int Hk, int Hv, int dk, int dv, int K, ddt_dtype in);
cudaError_t launch_gdn_tc(int L, int B, int N, int Hk, int Hv, int K, ddt_dtype in, ddt_dtype out, const void* x,
                          const void* conv_w, const void* conv_state, const float* beta, const float* decay,
                          const float* S, const int32_t* parent, const int32_t* n_nodes, void* o, int32_t* status,
                          cudaStream_t st);
size_t gdn_smem_bytes(int N, int dk, int dv);
// every node's branch-local state, the literal way (debugging aid for small trees)
cudaError_t launch_gdn_states(int L, int B, int N, int Hk, int Hv, int dk, int dv, int K, ddt_dtype in,
                              const void* x, const void* conv_w, const void* conv_state, const float* beta,
                              const float* decay, const float* S, const int32_t* parent, const int32_t* n_nodes,
                              float* S_node, cudaStream_t st);
cudaError_t launch_gdn_tree(int L, int B, int N, int Hk, int Hv, int dk, int dv, int K, ddt_dtype in,
                            ddt_dtype out, const void* x, const void* conv_w, const void* conv_state,
                            const float* beta, const float* decay, const float* S, const int32_t* parent,
                            const int32_t* n_nodes, void* o, int32_t* status, cudaStream_t st);

cudaError_t launch_commit(int B, int N, int A, int La, int Hkv, int d, int Pcap, ddt_dtype kv_dtype,
                          const void* k_tree, const void* v_tree, void* k_cache, void* v_cache, int Lg, int Hk,
                          int Hv, int dk, int dv, int K, ddt_dtype x_dtype, const void* x, const void* conv_w,
                          const float* beta, const float* decay, float* S, void* conv_state,
                          const int32_t* acc_nodes, const int32_t* acc_len, int32_t* prefix_len, int32_t* src_row,
                          int32_t* dst_pos, int32_t* status, const AttnPaging* paging, cudaStream_t st);

}  // namespace ddt
