// api.cu -- the extern "C" entry points of ddt.h: host-side argument checks, then
// stream-ordered kernel launches.  No device memory is allocated here and no host
// synchronisation happens; data errors found on the device go to the status words.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>

#include "ddt.h"
#include "kernels.h"

using namespace ddt;

namespace ddt {
static std::atomic<uint64_t> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace ddt

namespace {

inline ddt_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return DDT_OK;
    if (e == cudaErrorInvalidValue) return DDT_ERR_UNSUPPORTED;
    return DDT_ERR_CUDA;
}
inline bool dtype_ok(ddt_dtype t) { return t == DDT_F32 || t == DDT_BF16; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

const char* ddt_status_string(ddt_status s) {
    switch (s) {
        case DDT_OK: return "ok";
        case DDT_ERR_INVALID_ARG: return "invalid argument";
        case DDT_ERR_UNSUPPORTED: return "unsupported size or dtype combination";
        case DDT_ERR_CAPACITY: return "cache capacity exceeded";
        case DDT_ERR_CUDA: return "CUDA launch error";
        case DDT_ERR_TIMEOUT: return "bounded device wait gave up";
        case DDT_ERR_NONFINITE: return "non-finite logits";
        case DDT_ERR_TREE: return "malformed tree";
    }
    return "unknown status";
}

const char* ddt_version(void) { return "ddt 0.1 sm_103a"; }

uint64_t ddt_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

ddt_status ddt_wait_selftest(int32_t* status, ddt_stream_t stream) {
    if (!status) return DDT_ERR_INVALID_ARG;
    return launch_wait_selftest(status, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? DDT_OK
                                                                                            : DDT_ERR_CUDA;
}

// ------------------------------------------------------------------------- build
size_t ddt_build_tree_workspace(int B, int D, int V, int top_k) {
    if (B < 1 || D < 1 || V < 1 || top_k < 1) return 0;
    return build_ws_bytes(B, D, V, top_k);
}

ddt_status ddt_build_tree(int B, int D, int V, int top_k, int budget, ddt_dtype dtype, const void* draft_logits,
                          const int32_t* root_token, const int32_t* prefix_len, int32_t* token, int32_t* parent,
                          int32_t* depth, int32_t* position, int32_t* n_nodes, uint32_t* anc, double* score,
                          int32_t* status, void* workspace, size_t ws_bytes, ddt_stream_t stream) {
    if (B < 1 || D < 1 || V < 1 || top_k < 1 || budget < 0 || !dtype_ok(dtype)) return DDT_ERR_INVALID_ARG;
    if (D > kMaxDepth || top_k > kMaxTopK || top_k > V || budget > kMaxBudget) return DDT_ERR_UNSUPPORTED;
    if (!draft_logits || !root_token || !prefix_len || !token || !parent || !depth || !position || !n_nodes ||
        !anc || !status || !workspace)
        return DDT_ERR_INVALID_ARG;
    if (ws_bytes < build_ws_bytes(B, D, V, top_k) || !aligned16(workspace)) return DDT_ERR_INVALID_ARG;
    if (build_tree_smem(D, top_k, budget) > 200 * 1024) return DDT_ERR_UNSUPPORTED;
    return from_cuda(launch_build_tree(B, D, V, top_k, budget, dtype, draft_logits, root_token, prefix_len, token,
                                       parent, depth, position, n_nodes, anc, score, status, workspace,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------------ attention
size_t ddt_tree_attn_workspace(int n_layers, int B, int N, int Hq, int Hkv, int d, int Pcap) {
    if (n_layers < 1 || B < 1 || N < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Pcap < 0) return 0;
    return attn_tc_ws_bytes(n_layers, B, N, Hq, Hkv, d, Pcap);
}

ddt_status ddt_tree_attn(int n_layers, int B, int N, int Hq, int Hkv, int d, int Pcap, ddt_dtype in_dtype,
                         ddt_dtype out_dtype, const void* q, const void* k_tree, const void* v_tree,
                         const void* k_cache, const void* v_cache, const int32_t* prefix_len, const int32_t* n_nodes,
                         const uint32_t* anc, float scale, void* o, int32_t* status, void* workspace,
                         size_t ws_bytes, ddt_stream_t stream) {
    if (n_layers < 1 || B < 1 || N < 1 || Hq < 1 || Hkv < 1 || Pcap < 0 || !dtype_ok(in_dtype) ||
        !dtype_ok(out_dtype))
        return DDT_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return DDT_ERR_INVALID_ARG;
    if (N > kMaxRows || (d != 64 && d != 128 && d != 256)) return DDT_ERR_UNSUPPORTED;
    if (!q || !k_tree || !v_tree || (Pcap > 0 && (!k_cache || !v_cache)) || !prefix_len || !n_nodes || !anc || !o ||
        !status)
        return DDT_ERR_INVALID_ARG;
    // bf16 with a compiled head size runs on the tensor cores; fp32 on the CUDA cores
    if (attn_tc_supported(d, in_dtype)) {
        if (!workspace || ws_bytes < attn_tc_ws_bytes(n_layers, B, N, Hq, Hkv, d, Pcap) || !aligned16(workspace))
            return DDT_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k_tree) || !aligned16(v_tree) || !aligned16(o) ||
            (Pcap > 0 && (!aligned16(k_cache) || !aligned16(v_cache))))
            return DDT_ERR_INVALID_ARG;
        return from_cuda(launch_attn_tc(n_layers, B, N, Hq, Hkv, d, Pcap, out_dtype, q, k_tree, v_tree, k_cache,
                                        v_cache, prefix_len, n_nodes, anc, scale, o, status, workspace, ws_bytes,
                                        reinterpret_cast<cudaStream_t>(stream)));
    }
    return from_cuda(launch_attn_simt(n_layers, B, N, Hq, Hkv, d, Pcap, in_dtype, out_dtype, q, k_tree, v_tree,
                                      k_cache, v_cache, prefix_len, n_nodes, anc, scale, o, status,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

static bool page_rows_ok(int r) { return r >= 8 && r <= 4096 && (r >= 64 ? r % 64 == 0 : 64 % r == 0); }

size_t ddt_tree_attn_paged_workspace(int n_layers, int B, int N, int Hq, int Hkv, int d, int page_size,
                                     int max_pages) {
    if (!page_rows_ok(page_size) || max_pages < 1) return 0;
    return ddt_tree_attn_workspace(n_layers, B, N, Hq, Hkv, d, page_size * max_pages);
}

ddt_status ddt_tree_attn_paged(int n_layers, int B, int N, int Hq, int Hkv, int d, int page_size, int num_pages,
                               int max_pages, ddt_dtype in_dtype, ddt_dtype out_dtype, const void* q,
                               const void* k_tree, const void* v_tree, const void* k_pages, const void* v_pages,
                               const int32_t* block_table, const int32_t* prefix_len, const int32_t* n_nodes,
                               const uint32_t* anc, float scale, void* o, int32_t* status, void* workspace,
                               size_t ws_bytes, ddt_stream_t stream) {
    if (n_layers < 1 || B < 1 || N < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || num_pages < 1 || max_pages < 1 ||
        !dtype_ok(in_dtype) || !dtype_ok(out_dtype))
        return DDT_ERR_INVALID_ARG;
    if (!page_rows_ok(page_size) || (long)page_size * max_pages > (1L << 30)) return DDT_ERR_UNSUPPORTED;
    if (N > kMaxRows || !attn_tc_supported(d, in_dtype)) return DDT_ERR_UNSUPPORTED;
    if (!q || !k_tree || !v_tree || !k_pages || !v_pages || !block_table || !prefix_len || !n_nodes || !anc || !o ||
        !status)
        return DDT_ERR_INVALID_ARG;
    const AttnPaging pg{page_size, num_pages, max_pages, block_table};
    if (!workspace || ws_bytes < attn_tc_ws_bytes(n_layers, B, N, Hq, Hkv, d, page_size * max_pages) ||
        !aligned16(workspace))
        return DDT_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_tree) || !aligned16(v_tree) || !aligned16(o) || !aligned16(k_pages) ||
        !aligned16(v_pages))
        return DDT_ERR_INVALID_ARG;
    return from_cuda(launch_attn_tc_paged(n_layers, B, N, Hq, Hkv, d, pg, out_dtype, q, k_tree, v_tree, k_pages,
                                          v_pages, prefix_len, n_nodes, anc, scale, o, status, workspace, ws_bytes,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

ddt_status ddt_rope_tree(int n_layers, int B, int N, int Hq, int Hkv, int d, int rot_dim, double theta,
                         ddt_dtype dtype, const int32_t* position, const int32_t* n_nodes, void* q, void* k_tree,
                         ddt_stream_t stream) {
    if (n_layers < 1 || B < 1 || N < 1 || Hq < 1 || Hkv < 1 || d < 2 || !dtype_ok(dtype)) return DDT_ERR_INVALID_ARG;
    if (rot_dim < 2 || rot_dim > d || rot_dim % 2 != 0 || !(theta > 1.0)) return DDT_ERR_INVALID_ARG;
    if (!position || !n_nodes || !k_tree) return DDT_ERR_INVALID_ARG;  // q NULL: rotate the keys only
    if (B > 65535) return DDT_ERR_UNSUPPORTED;
    return from_cuda(launch_rope_tree(n_layers, B, N, Hq, Hkv, d, rot_dim, theta, dtype, position, n_nodes, q, k_tree,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

// Rotary variants: q is taken before rotary embedding and rotated while the attention
// kernel stages it; the cos/sin table of every row's position goes to the end of the
// workspace (after the ddt_tree_attn(_paged)_workspace bytes).
static size_t rope_table_offset(size_t base) { return (base + 255) & ~(size_t)255; }

static ddt_status rope_args_ok(int d, ddt_dtype in_dtype, int rot_dim, double theta, const int32_t* position) {
    if (!position || rot_dim < 16 || rot_dim > d || rot_dim % 16 != 0 || !(theta > 1.0)) return DDT_ERR_INVALID_ARG;
    if (in_dtype != DDT_BF16 || (d != 128 && d != 256)) return DDT_ERR_UNSUPPORTED;
    return DDT_OK;
}

ddt_status ddt_tree_attn_rope(int n_layers, int B, int N, int Hq, int Hkv, int d, int Pcap, ddt_dtype in_dtype,
                              ddt_dtype out_dtype, const void* q, const void* k_tree, const void* v_tree,
                              const void* k_cache, const void* v_cache, const int32_t* prefix_len,
                              const int32_t* n_nodes, const uint32_t* anc, const int32_t* position, int rot_dim,
                              double theta, float scale, void* o, int32_t* status, void* workspace, size_t ws_bytes,
                              ddt_stream_t stream) {
    if (n_layers < 1 || B < 1 || N < 1 || Hq < 1 || Hkv < 1 || Pcap < 0 || Hq % Hkv != 0 || !dtype_ok(in_dtype) ||
        !dtype_ok(out_dtype))
        return DDT_ERR_INVALID_ARG;
    if (N > kMaxRows || B > 65535) return DDT_ERR_UNSUPPORTED;
    const ddt_status ra = rope_args_ok(d, in_dtype, rot_dim, theta, position);
    if (ra != DDT_OK) return ra;
    if (!q || !k_tree || !v_tree || (Pcap > 0 && (!k_cache || !v_cache)) || !prefix_len || !n_nodes || !anc || !o ||
        !status || !workspace || !aligned16(workspace))
        return DDT_ERR_INVALID_ARG;
    const size_t base = attn_tc_ws_bytes(n_layers, B, N, Hq, Hkv, d, Pcap);
    const size_t off = rope_table_offset(base);
    if (ws_bytes < off + sizeof(float) * (size_t)B * N * rot_dim) return DDT_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_tree) || !aligned16(v_tree) || !aligned16(o) ||
        (Pcap > 0 && (!aligned16(k_cache) || !aligned16(v_cache))))
        return DDT_ERR_INVALID_ARG;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* table = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + off);
    cudaError_t e = launch_rope_table(B, N, rot_dim, theta, position, n_nodes, table, st);
    if (e != cudaSuccess) return from_cuda(e);
    const AttnRope rope{rot_dim, table};
    return from_cuda(launch_attn_tc(n_layers, B, N, Hq, Hkv, d, Pcap, out_dtype, q, k_tree, v_tree, k_cache, v_cache,
                                    prefix_len, n_nodes, anc, scale, o, status, workspace, base, st, &rope));
}

ddt_status ddt_tree_attn_paged_rope(int n_layers, int B, int N, int Hq, int Hkv, int d, int page_size, int num_pages,
                                    int max_pages, ddt_dtype in_dtype, ddt_dtype out_dtype, const void* q,
                                    const void* k_tree, const void* v_tree, const void* k_pages, const void* v_pages,
                                    const int32_t* block_table, const int32_t* prefix_len, const int32_t* n_nodes,
                                    const uint32_t* anc, const int32_t* position, int rot_dim, double theta,
                                    float scale, void* o, int32_t* status, void* workspace, size_t ws_bytes,
                                    ddt_stream_t stream) {
    if (n_layers < 1 || B < 1 || N < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || num_pages < 1 || max_pages < 1 ||
        !dtype_ok(in_dtype) || !dtype_ok(out_dtype))
        return DDT_ERR_INVALID_ARG;
    if (!page_rows_ok(page_size) || (long)page_size * max_pages > (1L << 30)) return DDT_ERR_UNSUPPORTED;
    if (N > kMaxRows || B > 65535) return DDT_ERR_UNSUPPORTED;
    const ddt_status ra = rope_args_ok(d, in_dtype, rot_dim, theta, position);
    if (ra != DDT_OK) return ra;
    if (!q || !k_tree || !v_tree || !k_pages || !v_pages || !block_table || !prefix_len || !n_nodes || !anc || !o ||
        !status || !workspace || !aligned16(workspace))
        return DDT_ERR_INVALID_ARG;
    const size_t base = attn_tc_ws_bytes(n_layers, B, N, Hq, Hkv, d, page_size * max_pages);
    const size_t off = rope_table_offset(base);
    if (ws_bytes < off + sizeof(float) * (size_t)B * N * rot_dim) return DDT_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_tree) || !aligned16(v_tree) || !aligned16(o) || !aligned16(k_pages) ||
        !aligned16(v_pages))
        return DDT_ERR_INVALID_ARG;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* table = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + off);
    cudaError_t e = launch_rope_table(B, N, rot_dim, theta, position, n_nodes, table, st);
    if (e != cudaSuccess) return from_cuda(e);
    const AttnPaging pg{page_size, num_pages, max_pages, block_table};
    const AttnRope rope{rot_dim, table};
    return from_cuda(launch_attn_tc_paged(n_layers, B, N, Hq, Hkv, d, pg, out_dtype, q, k_tree, v_tree, k_pages,
                                          v_pages, prefix_len, n_nodes, anc, scale, o, status, workspace, base, st,
                                          &rope));
}

// ------------------------------------------------------------------------------ GDN
size_t ddt_tree_gdn_workspace(int n_layers, int B, int N, int Hk, int Hv, int dk, int dv) {
    (void)n_layers; (void)B; (void)N; (void)Hk; (void)Hv; (void)dk; (void)dv;
    return 256;
}

ddt_status ddt_tree_gdn(int n_layers, int B, int N, int Hk, int Hv, int dk, int dv, int conv_k, ddt_dtype in_dtype,
                        ddt_dtype out_dtype, const void* x, const void* conv_w, const void* conv_state,
                        const float* beta, const float* decay, const float* S, const int32_t* parent,
                        const int32_t* n_nodes, void* o, float* S_node_debug, int32_t* status, void* workspace,
                        size_t ws_bytes, ddt_stream_t stream) {
    (void)workspace; (void)ws_bytes;
    if (n_layers < 1 || B < 1 || N < 1 || Hk < 1 || Hv < 1 || Hv % Hk != 0 || conv_k < 1 || !dtype_ok(in_dtype) ||
        !dtype_ok(out_dtype))
        return DDT_ERR_INVALID_ARG;
    const bool dims = (dk == 32 && dv == 32) || (dk == 64 && dv == 64) || (dk == 128 && dv == 128) ||
                      (dk == 64 && dv == 128) || (dk == 128 && dv == 64);
    if (!dims || conv_k > 8 || N > kGdnMaxNodes || gdn_smem_bytes(N, dk, dv) > 227 * 1024) return DDT_ERR_UNSUPPORTED;
    if (!x || !conv_w || (conv_k > 1 && !conv_state) || !beta || !decay || !S || !parent || !n_nodes || !o ||
        !status || !aligned16(S))
        return DDT_ERR_INVALID_ARG;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    // head size 128: dense part on the tensor cores (its TMA row loads want x and the conv
    // state 16-byte aligned); other sizes on the CUDA cores
    if (gdn_tc_supported(N, Hk, Hv, dk, dv, conv_k, in_dtype) && aligned16(x) && (conv_k == 1 || aligned16(conv_state)))
        e = launch_gdn_tc(n_layers, B, N, Hk, Hv, conv_k, in_dtype, out_dtype, x, conv_w, conv_state, beta, decay, S,
                          parent, n_nodes, o, status, st);
    else
        e = launch_gdn_tree(n_layers, B, N, Hk, Hv, dk, dv, conv_k, in_dtype, out_dtype, x, conv_w, conv_state, beta,
                            decay, S, parent, n_nodes, o, status, st);
    if (e == cudaSuccess && S_node_debug)
        e = launch_gdn_states(n_layers, B, N, Hk, Hv, dk, dv, conv_k, in_dtype, x, conv_w, conv_state, beta, decay,
                              S, parent, n_nodes, S_node_debug, st);
    return from_cuda(e);
}

// ----------------------------------------------------------------------------- walk
size_t ddt_walk_accept_workspace(int B, int N, int V) {
    if (B < 1 || N < 1 || V < 1) return 0;
    return walk_ws_bytes(B, N, V);
}

static ddt_status walk_accept(int B, int N, int V, int max_accept, ddt_dtype dtype, const void* target_logits,
                              int32_t* target_argmax, const int32_t* token, const int32_t* parent,
                              const int32_t* n_nodes, int32_t* acc_nodes, int32_t* acc_len, int32_t* bonus,
                              int32_t* emitted, int32_t* n_emitted, int32_t* status, void* workspace, size_t ws_bytes,
                              int flat, ddt_stream_t stream) {
    if (B < 1 || N < 1 || V < 1 || max_accept < 0 || !dtype_ok(dtype)) return DDT_ERR_INVALID_ARG;
    if (N > kMaxRows) return DDT_ERR_UNSUPPORTED;
    if (!target_argmax || !token || !parent || !n_nodes || !acc_nodes || !acc_len || !bonus || !emitted ||
        !n_emitted || !status)
        return DDT_ERR_INVALID_ARG;
    if (target_logits && (!workspace || ws_bytes < walk_ws_bytes(B, N, V) || !aligned16(workspace)))
        return DDT_ERR_INVALID_ARG;
    return from_cuda(launch_walk(B, N, V, max_accept + 1, dtype, target_logits, target_argmax, token, parent, n_nodes,
                                 acc_nodes, acc_len, bonus, emitted, n_emitted, status, workspace, flat,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

ddt_status ddt_walk_accept(int B, int N, int V, int max_accept, ddt_dtype dtype, const void* target_logits,
                           int32_t* target_argmax, const int32_t* token, const int32_t* parent,
                           const int32_t* n_nodes, int32_t* acc_nodes, int32_t* acc_len, int32_t* bonus,
                           int32_t* emitted, int32_t* n_emitted, int32_t* status, void* workspace, size_t ws_bytes,
                           ddt_stream_t stream) {
    return walk_accept(B, N, V, max_accept, dtype, target_logits, target_argmax, token, parent, n_nodes, acc_nodes,
                       acc_len, bonus, emitted, n_emitted, status, workspace, ws_bytes, 0, stream);
}

ddt_status ddt_walk_accept_flat(int B, int N, int V, int max_accept, ddt_dtype dtype, const void* target_logits,
                                int32_t* target_argmax, const int32_t* token, const int32_t* parent,
                                const int32_t* n_nodes, int32_t* acc_nodes, int32_t* acc_len, int32_t* bonus,
                                int32_t* emitted, int32_t* n_emitted, int32_t* status, void* workspace,
                                size_t ws_bytes, ddt_stream_t stream) {
    return walk_accept(B, N, V, max_accept, dtype, target_logits, target_argmax, token, parent, n_nodes, acc_nodes,
                       acc_len, bonus, emitted, n_emitted, status, workspace, ws_bytes, 1, stream);
}

size_t ddt_walk_accept_sample_workspace(int B, int N, int V) {
    if (B < 1 || N < 1 || V < 1) return 0;
    return walk_sample_ws_bytes(B, N, V);
}

ddt_status ddt_walk_accept_sample(int B, int N, int V, int max_accept, int max_children, float temperature,
                                  ddt_dtype dtype, const void* target_logits, const float* uniforms,
                                  const int32_t* token, const int32_t* parent, const int32_t* n_nodes,
                                  int32_t* acc_nodes, int32_t* acc_len, int32_t* bonus, int32_t* emitted,
                                  int32_t* n_emitted, int32_t* status, void* workspace, size_t ws_bytes,
                                  ddt_stream_t stream) {
    if (B < 1 || N < 1 || V < 1 || max_accept < 0 || max_children < 1 || !dtype_ok(dtype)) return DDT_ERR_INVALID_ARG;
    // T > 0 with a finite fp32 reciprocal (the kernels scale by 1/T)
    if (!(temperature > 0.0f) || !(1.0f / temperature < INFINITY) || !(temperature < INFINITY))
        return DDT_ERR_INVALID_ARG;
    if (N > kMaxRows || B > 65535 || max_accept > kMaxAccept || max_children > kMaxTopK) return DDT_ERR_UNSUPPORTED;
    if (!target_logits || !uniforms || !token || !parent || !n_nodes || !acc_nodes || !acc_len || !bonus ||
        !emitted || !n_emitted || !status)
        return DDT_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < walk_sample_ws_bytes(B, N, V) || !aligned16(workspace)) return DDT_ERR_INVALID_ARG;
    return from_cuda(launch_walk_sample(B, N, V, max_accept + 1, max_children, temperature, dtype, target_logits,
                                        uniforms, token, parent, n_nodes, acc_nodes, acc_len, bonus, emitted,
                                        n_emitted, status, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------------------- commit
ddt_status ddt_commit(int B, int N, int A, int n_attn_layers, int Hkv, int d, int Pcap, ddt_dtype kv_dtype,
                      const void* k_tree, const void* v_tree, void* k_cache, void* v_cache, int n_gdn_layers, int Hk,
                      int Hv, int dk, int dv, int conv_k, ddt_dtype x_dtype, const void* x, const void* conv_w,
                      const float* beta, const float* decay, float* S, void* conv_state, const int32_t* acc_nodes,
                      const int32_t* acc_len, int32_t* prefix_len, int32_t* src_row, int32_t* dst_pos,
                      int32_t* status, ddt_stream_t stream) {
    if (B < 1 || N < 1 || A < 1 || n_attn_layers < 0 || n_gdn_layers < 0) return DDT_ERR_INVALID_ARG;
    if (A > kMaxAccept + 1) return DDT_ERR_UNSUPPORTED;
    if (!acc_nodes || !acc_len || !prefix_len || !src_row || !dst_pos || !status) return DDT_ERR_INVALID_ARG;
    if (n_attn_layers > 0) {
        if (Hkv < 1 || d < 1 || Pcap < 1 || !dtype_ok(kv_dtype) || !k_tree || !v_tree || !k_cache || !v_cache)
            return DDT_ERR_INVALID_ARG;
    }
    if (n_gdn_layers > 0) {
        if (Hk < 1 || Hv < 1 || Hv % Hk != 0 || conv_k < 1 || conv_k > 8 || !dtype_ok(x_dtype) || !x || !conv_w ||
            !beta || !decay || !S || (conv_k > 1 && !conv_state) || !aligned16(S))
            return DDT_ERR_INVALID_ARG;
        const bool dims = (dk == 32 && dv == 32) || (dk == 64 && dv == 64) || (dk == 128 && dv == 128) ||
                          (dk == 64 && dv == 128) || (dk == 128 && dv == 64);
        if (!dims) return DDT_ERR_UNSUPPORTED;
    }
    return from_cuda(launch_commit(B, N, A, n_attn_layers, Hkv, d, Pcap, kv_dtype, k_tree, v_tree, k_cache, v_cache,
                                   n_gdn_layers, Hk, Hv, dk, dv, conv_k, x_dtype, x, conv_w, beta, decay, S,
                                   conv_state, acc_nodes, acc_len, prefix_len, src_row, dst_pos, status, nullptr,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

ddt_status ddt_commit_paged(int B, int N, int A, int n_attn_layers, int Hkv, int d, int page_size, int num_pages,
                            int max_pages, const int32_t* block_table, ddt_dtype kv_dtype, const void* k_tree,
                            const void* v_tree, void* k_pages, void* v_pages, int n_gdn_layers, int Hk, int Hv, int dk,
                            int dv, int conv_k, ddt_dtype x_dtype, const void* x, const void* conv_w,
                            const float* beta, const float* decay, float* S, void* conv_state,
                            const int32_t* acc_nodes, const int32_t* acc_len, int32_t* prefix_len, int32_t* src_row,
                            int32_t* dst_pos, int32_t* status, ddt_stream_t stream) {
    if (n_attn_layers < 1 || !block_table || num_pages < 1 || max_pages < 1) return DDT_ERR_INVALID_ARG;
    if (!page_rows_ok(page_size) || (long)page_size * max_pages > (1L << 30)) return DDT_ERR_UNSUPPORTED;
    if (B < 1 || N < 1 || A < 1 || n_gdn_layers < 0) return DDT_ERR_INVALID_ARG;
    if (A > kMaxAccept + 1) return DDT_ERR_UNSUPPORTED;
    if (!acc_nodes || !acc_len || !prefix_len || !src_row || !dst_pos || !status) return DDT_ERR_INVALID_ARG;
    if (Hkv < 1 || d < 1 || !dtype_ok(kv_dtype) || !k_tree || !v_tree || !k_pages || !v_pages)
        return DDT_ERR_INVALID_ARG;
    if (n_gdn_layers > 0) {
        if (Hk < 1 || Hv < 1 || Hv % Hk != 0 || conv_k < 1 || conv_k > 8 || !dtype_ok(x_dtype) || !x || !conv_w ||
            !beta || !decay || !S || (conv_k > 1 && !conv_state) || !aligned16(S))
            return DDT_ERR_INVALID_ARG;
        const bool dims = (dk == 32 && dv == 32) || (dk == 64 && dv == 64) || (dk == 128 && dv == 128) ||
                          (dk == 64 && dv == 128) || (dk == 128 && dv == 64);
        if (!dims) return DDT_ERR_UNSUPPORTED;
    }
    const AttnPaging pg{page_size, num_pages, max_pages, block_table};
    return from_cuda(launch_commit(B, N, A, n_attn_layers, Hkv, d, page_size * max_pages, kv_dtype, k_tree, v_tree,
                                   k_pages, v_pages, n_gdn_layers, Hk, Hv, dk, dv, conv_k, x_dtype, x, conv_w, beta,
                                   decay, S, conv_state, acc_nodes, acc_len, prefix_len, src_row, dst_pos, status, &pg,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
