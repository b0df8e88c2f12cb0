// commit.cu -- ddt_commit: copy only the accepted path into the committed buffers.
//
// "DDTree on vLLM: candid research notes", sections "Why hybrid attention makes it hard"
// and "Where the next step is": once a path is accepted, only that path may be copied
// back into the contiguous KV and recurrent buffers (an explicit accepted-branch commit
// with first-class node and parent ids).  "From Tree-Based Speculative Decoding to
// Drafter Training", section "The Architecture of DDTree": the KV cache is compacted to
// the accepted path's entries.
//
//   k_commit_kv     grid (A, La*Hkv, B): 16-byte vector copy of one tree row into the
//                   cache at prefix_len + j.
//   k_commit_gdn    grid (Hv, B, Lg): the committed state (dv x dk fp32) is held in
//                   registers (two threads per row), advanced along the accepted path
//                   (<= A rank-one delta steps) and written back in place: one HBM read
//                   and one write.
//   k_commit_conv   grid (Lg, B): last K-1 raw inputs of [conv state ; path inputs].
//   k_commit_final  prefix_len, commit indices and status (runs last: the kernels above
//                   read the old prefix_len).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace ddt {

// Paged caches: position p of request b is row p % page_rows of physical page
// bt[b][p / page_rows] (bt == nullptr: contiguous caches).
struct KvPages {
    const int32_t* bt;
    int page_rows, num_pages, max_pages;
};

// A request's commit is valid when its accepted path is well formed and fits (and, paged,
// every page it writes exists).  Every commit kernel evaluates the same check.
__device__ __forceinline__ int commit_check(int b, int N, int A, int cap_check, int Pcap,
                                            const int32_t* acc_nodes, const int32_t* acc_len,
                                            const int32_t* prefix_len, const KvPages& pg) {
    const int a = acc_len[b];
    if (a < 0 || a + 1 > A) return DDT_ERR_INVALID_ARG;
    for (int j = 0; j <= a; ++j) {
        const int r = acc_nodes[(long)b * A + j];
        if (r < 0 || r >= N) return DDT_ERR_TREE;
    }
    if (cap_check && (prefix_len[b] < 0 || prefix_len[b] + a + 1 > Pcap)) return DDT_ERR_CAPACITY;
    if (cap_check && pg.bt)
        for (int j = 0; j <= a; ++j) {
            const int phys = pg.bt[(long)b * pg.max_pages + (prefix_len[b] + j) / pg.page_rows];
            if (phys < 0 || phys >= pg.num_pages) return DDT_ERR_INVALID_ARG;
        }
    return DDT_OK;
}

template <typename T>
__global__ void k_commit_kv(int B, int N, int A, int Hkv, int d, int Pcap, int vec, const T* __restrict__ k_tree,
                            const T* __restrict__ v_tree, T* __restrict__ k_cache, T* __restrict__ v_cache,
                            const int32_t* __restrict__ acc_nodes, const int32_t* __restrict__ acc_len,
                            const int32_t* __restrict__ prefix_len, const KvPages pg) {
    const int j = blockIdx.x, lg = blockIdx.y, b = blockIdx.z;
    const int l = lg / Hkv, g = lg % Hkv;
    __shared__ int s_ok;
    if (threadIdx.x == 0) s_ok = commit_check(b, N, A, 1, Pcap, acc_nodes, acc_len, prefix_len, pg) == DDT_OK;
    __syncthreads();
    if (!s_ok || j > acc_len[b]) return;
    const int src = acc_nodes[(long)b * A + j];
    const long lb = (long)l * B + b;
    const long so = ((lb * N + src) * Hkv + g) * (long)d;
    const int pos = prefix_len[b] + j;
    long dof;
    if (pg.bt) {
        const long phys = pg.bt[(long)b * pg.max_pages + pos / pg.page_rows];
        dof = ((((long)l * pg.num_pages + phys) * Hkv + g) * pg.page_rows + pos % pg.page_rows) * d;
    } else {
        dof = ((lb * Hkv + g) * (long)Pcap + pos) * d;
    }
    if (vec) {
        const int nv = d * (int)sizeof(T) / 16;
        for (int e = threadIdx.x; e < nv; e += blockDim.x) {
            reinterpret_cast<uint4*>(k_cache + dof)[e] = reinterpret_cast<const uint4*>(k_tree + so)[e];
            reinterpret_cast<uint4*>(v_cache + dof)[e] = reinterpret_cast<const uint4*>(v_tree + so)[e];
        }
    } else {
        for (int e = threadIdx.x; e < d; e += blockDim.x) {
            k_cache[dof + e] = k_tree[so + e];
            v_cache[dof + e] = v_tree[so + e];
        }
    }
}

__device__ __forceinline__ float silu_c(float z) { return z / (1.f + __expf(-z)); }

// One CTA per (value head, request, layer), 2 threads per state row on average (DV rows):
// the state lives in registers, DK/2 entries a thread.  Prologue: conv + SiLU of the k and v
// channels of every accepted node (all loads in flight together), k norms and gates into
// shared memory.  Then the a + 1 delta steps need no barrier: each row's S k is eight
// partial dots joined by three shuffles, and the rank-one update is in registers.
template <typename Tx, int DK, int DV>
__global__ void __launch_bounds__(2 * DV, 2) k_commit_gdn(int B, int N, int A, int Hk, int Hv, int K, int cap_check,
                                                       int Pcap, const Tx* __restrict__ x,
                                                       const Tx* __restrict__ conv_w,
                                                       const Tx* __restrict__ conv_state,
                                                       const float* __restrict__ beta,
                                                       const float* __restrict__ decay, float* __restrict__ S,
                                                       const int32_t* __restrict__ acc_nodes,
                                                       const int32_t* __restrict__ acc_len,
                                                       const int32_t* __restrict__ prefix_len, const KvPages pg) {
    constexpr int kT = 2 * DV, kH = DK / 2;
    extern __shared__ __align__(16) float sm[];
    float* s_k = sm;                 // [A][DK]  normalised k of each accepted node
    float* s_v = s_k + A * DK;       // [A][DV]
    float* s_g = s_v + A * DV;       // [A][2]   decay, beta
    __shared__ int s_ok;
    const int h = blockIdx.x, b = blockIdx.y, l = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_ok = commit_check(b, N, A, cap_check, Pcap, acc_nodes, acc_len, prefix_len, pg) == DDT_OK;
    __syncthreads();
    if (!s_ok) return;
    const int a = acc_len[b];
    const int C = 2 * Hk * DK + Hv * DV;
    const int g = h / (Hv / Hk);
    const long lb = (long)l * B + b;
    const int32_t* path = acc_nodes + (long)b * A;
    const Tx* xb = x + lb * N * C;
    const Tx* cs = conv_state + lb * (K - 1) * C;
    const Tx* wl = conv_w + (long)l * C * K;

    // conv + SiLU of the k and v channels along the accepted path
    for (int e = tid; e < DK + DV; e += kT) {
        const int c = (e < DK) ? (Hk * DK + g * DK + e) : (2 * Hk * DK + h * DV + e - DK);
        float w[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) w[q] = q < K ? to_f32(wl[(long)c * K + q]) : 0.f;
#pragma unroll 2
        for (int t = 0; t <= a; ++t) {
            float acc = 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (q < K) {
                    const int back = K - 1 - q;
                    const float in = (back <= t) ? to_f32(xb[(long)path[t - back] * C + c])
                                                 : to_f32(cs[(long)(K - 1 - (back - t)) * C + c]);
                    acc = fmaf(w[q], in, acc);
                }
            }
            if (e < DK) s_k[t * DK + e] = silu_c(acc);
            else s_v[t * DV + e - DK] = silu_c(acc);
        }
    }
    for (int t = tid; t <= a; t += kT) {
        s_g[2 * t] = decay[(lb * N + path[t]) * Hv + h];
        s_g[2 * t + 1] = beta[(lb * N + path[t]) * Hv + h];
    }
    __syncthreads();
    // the state rows (their loads overlap the k normalisation).  A warp holds 16 rows; the
    // eight lanes of row group rg = lane / 8 share rows 16 warp + rg + 4 i (i < 4) and lane
    // sub = lane % 8 takes 16-byte chunks sub + 8 m of each, so every load or store of the
    // warp covers four whole 128-byte row segments
    static_assert(DK % 32 == 0 && DV % 16 == 0, "state tile: 8 lanes x 16-byte chunks per row, 16 rows a warp");
    constexpr int kC = DK / 32;  // chunks a lane takes per row
    const int sub = lane & 7, rg = lane >> 3;
    float* Sg = S + (lb * Hv + h) * (long)DV * DK;
    float sr[kH];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < kC; ++m) {
            const float4 v4 =
                *reinterpret_cast<const float4*>(Sg + (long)(16 * warp + rg + 4 * i) * DK + 4 * (sub + 8 * m));
            sr[(i * kC + m) * 4] = v4.x;
            sr[(i * kC + m) * 4 + 1] = v4.y;
            sr[(i * kC + m) * 4 + 2] = v4.z;
            sr[(i * kC + m) * 4 + 3] = v4.w;
        }

    // k normalisation: one warp per node
    for (int t = warp; t <= a; t += kT / 32) {
        float ss = 0.f;
        for (int i = lane; i < DK; i += 32) ss = fmaf(s_k[t * DK + i], s_k[t * DK + i], ss);
        ss = warp_sum(ss);
        const float rk = rsqrtf(ss + 1e-6f);
        __syncwarp();
        for (int i = lane; i < DK; i += 32) s_k[t * DK + i] *= rk;
    }
    __syncthreads();

    for (int t = 0; t <= a; ++t) {
        const float* kt = s_k + t * DK;
        const float at = s_g[2 * t], bt = s_g[2 * t + 1];
        float kv[kC * 4];
#pragma unroll
        for (int m = 0; m < kC; ++m) {
            const float4 k4 = *reinterpret_cast<const float4*>(kt + 4 * (sub + 8 * m));
            kv[4 * m] = k4.x;
            kv[4 * m + 1] = k4.y;
            kv[4 * m + 2] = k4.z;
            kv[4 * m + 3] = k4.w;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float part = 0.f;
#pragma unroll
            for (int c = 0; c < kC * 4; ++c) part = fmaf(sr[i * kC * 4 + c], kv[c], part);
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            part += __shfl_xor_sync(0xffffffffu, part, 4);
            const float u = bt * (s_v[t * DV + 16 * warp + rg + 4 * i] - at * part);  // u = b (v - a S k^)
#pragma unroll
            for (int c = 0; c < kC * 4; ++c) sr[i * kC * 4 + c] = fmaf(at, sr[i * kC * 4 + c], u * kv[c]);  // S <- a S + u k^T
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < kC; ++m)
            *reinterpret_cast<float4*>(Sg + (long)(16 * warp + rg + 4 * i) * DK + 4 * (sub + 8 * m)) =
                make_float4(sr[(i * kC + m) * 4], sr[(i * kC + m) * 4 + 1], sr[(i * kC + m) * 4 + 2],
                            sr[(i * kC + m) * 4 + 3]);
}

template <typename Tx>
__global__ void k_commit_conv(int B, int N, int A, int C, int K, int cap_check, int Pcap, int vec,
                              const Tx* __restrict__ x, Tx* __restrict__ conv_state,
                              const int32_t* __restrict__ acc_nodes, const int32_t* __restrict__ acc_len,
                              const int32_t* __restrict__ prefix_len, const KvPages pg) {
    const int l = blockIdx.x, b = blockIdx.y;
    __shared__ int s_ok;
    if (threadIdx.x == 0) s_ok = commit_check(b, N, A, cap_check, Pcap, acc_nodes, acc_len, prefix_len, pg) == DDT_OK;
    __syncthreads();
    if (!s_ok) return;
    const int n = acc_len[b] + 1;
    const long lb = (long)l * B + b;
    Tx* cs = conv_state + lb * (K - 1) * C;
    const Tx* xb = x + lb * N * C;
    const int32_t* path = acc_nodes + (long)b * A;
    // new row r = entry r + n of [cs ; path rows]; each element is read before it is
    // rewritten (r + n > r, and one thread owns a column chunk across all rows)
    if (vec) {  // 16-byte chunks of a row
        const int nc = C * (int)sizeof(Tx) / 16;
        for (int q = threadIdx.x; q < nc; q += blockDim.x)
            for (int r = 0; r < K - 1; ++r) {
                const int src = r + n;
                const Tx* from = (src < K - 1) ? cs + (long)src * C : xb + (long)path[src - (K - 1)] * C;
                reinterpret_cast<uint4*>(cs + (long)r * C)[q] = reinterpret_cast<const uint4*>(from)[q];
            }
    } else {
        for (int c = threadIdx.x; c < C; c += blockDim.x)
            for (int r = 0; r < K - 1; ++r) {
                const int src = r + n;
                cs[(long)r * C + c] = (src < K - 1) ? cs[(long)src * C + c] : xb[(long)path[src - (K - 1)] * C + c];
            }
    }
}

__global__ void k_commit_final(int B, int N, int A, int cap_check, int Pcap, const int32_t* __restrict__ acc_nodes,
                               const int32_t* __restrict__ acc_len, int32_t* __restrict__ prefix_len,
                               int32_t* __restrict__ src_row, int32_t* __restrict__ dst_pos,
                               int32_t* __restrict__ status, const KvPages pg) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int st = commit_check(b, N, A, cap_check, Pcap, acc_nodes, acc_len, prefix_len, pg);
    const int P = prefix_len[b];
    const int a = acc_len[b];
    for (int j = 0; j < A; ++j) {
        const bool on = st == DDT_OK && j <= a;
        src_row[(long)b * A + j] = on ? acc_nodes[(long)b * A + j] : -1;
        dst_pos[(long)b * A + j] = on ? P + j : -1;
    }
    if (st == DDT_OK) prefix_len[b] = P + a + 1;
    status[b] = st;
}

template <typename Tx, int DK, int DV>
static cudaError_t commit_gdn_go(int B, int N, int A, int Lg, int Hk, int Hv, int K, int cap, int Pcap,
                                 const void* x, const void* w, const void* cs, const float* beta,
                                 const float* decay, float* S, const int32_t* an, const int32_t* al,
                                 const int32_t* pl, const KvPages& pg, cudaStream_t st) {
    const size_t smem = sizeof(float) * (size_t)A * (DK + DV + 2);
    cudaError_t e = cudaFuncSetAttribute(k_commit_gdn<Tx, DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    k_commit_gdn<Tx, DK, DV><<<counted(dim3(Hv, B, Lg)), 2 * DV, smem, st>>>(
        B, N, A, Hk, Hv, K, cap, Pcap, static_cast<const Tx*>(x), static_cast<const Tx*>(w),
        static_cast<const Tx*>(cs), beta, decay, S, an, al, pl, pg);
    return cudaGetLastError();
}

template <typename Tx>
static cudaError_t commit_gdn_dims(int dk, int dv, int B, int N, int A, int Lg, int Hk, int Hv, int K, int cap,
                                   int Pcap, const void* x, const void* w, const void* cs, const float* beta,
                                   const float* decay, float* S, const int32_t* an, const int32_t* al,
                                   const int32_t* pl, const KvPages& pg, cudaStream_t st) {
#define DDT_CG_CASE(P, Q)                                                                                        \
    if (dk == P && dv == Q)                                                                                      \
        return commit_gdn_go<Tx, P, Q>(B, N, A, Lg, Hk, Hv, K, cap, Pcap, x, w, cs, beta, decay, S, an, al, pl, pg, \
                                       st);
    DDT_CG_CASE(32, 32)
    DDT_CG_CASE(64, 64)
    DDT_CG_CASE(128, 128)
    DDT_CG_CASE(64, 128)
    DDT_CG_CASE(128, 64)
#undef DDT_CG_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_commit(int B, int N, int A, int La, int Hkv, int d, int Pcap, ddt_dtype kv_dtype,
                          const void* k_tree, const void* v_tree, void* k_cache, void* v_cache, int Lg, int Hk,
                          int Hv, int dk, int dv, int K, ddt_dtype x_dtype, const void* x, const void* conv_w,
                          const float* beta, const float* decay, float* S, void* conv_state,
                          const int32_t* acc_nodes, const int32_t* acc_len, int32_t* prefix_len, int32_t* src_row,
                          int32_t* dst_pos, int32_t* status, const AttnPaging* paging, cudaStream_t st) {
    cudaError_t e;
    const int cap = La > 0;
    const KvPages pg = paging ? KvPages{paging->block_table, paging->page_rows, paging->num_pages, paging->max_pages}
                              : KvPages{nullptr, 0, 0, 0};
    if (La > 0) {
        const size_t es = kv_dtype == DDT_BF16 ? 2 : 4;
        const int vec = ((d * es) % 16 == 0) && (reinterpret_cast<uintptr_t>(k_tree) % 16 == 0) &&
                        (reinterpret_cast<uintptr_t>(v_tree) % 16 == 0) &&
                        (reinterpret_cast<uintptr_t>(k_cache) % 16 == 0) &&
                        (reinterpret_cast<uintptr_t>(v_cache) % 16 == 0);
        dim3 grid(A, La * Hkv, B);
        if (kv_dtype == DDT_BF16)
            k_commit_kv<__nv_bfloat16><<<counted(grid), 64, 0, st>>>(
                B, N, A, Hkv, d, Pcap, vec, static_cast<const __nv_bfloat16*>(k_tree),
                static_cast<const __nv_bfloat16*>(v_tree), static_cast<__nv_bfloat16*>(k_cache),
                static_cast<__nv_bfloat16*>(v_cache), acc_nodes, acc_len, prefix_len, pg);
        else
            k_commit_kv<float><<<counted(grid), 64, 0, st>>>(B, N, A, Hkv, d, Pcap, vec, static_cast<const float*>(k_tree),
                                                    static_cast<const float*>(v_tree), static_cast<float*>(k_cache),
                                                    static_cast<float*>(v_cache), acc_nodes, acc_len, prefix_len, pg);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (Lg > 0) {
        const int C = 2 * Hk * dk + Hv * dv;
        const int cvec = ((C * (x_dtype == DDT_BF16 ? 2 : 4)) % 16 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(conv_state) % 16 == 0);
        if (x_dtype == DDT_BF16) {
            e = commit_gdn_dims<__nv_bfloat16>(dk, dv, B, N, A, Lg, Hk, Hv, K, cap, Pcap, x, conv_w, conv_state, beta,
                                               decay, S, acc_nodes, acc_len, prefix_len, pg, st);
            if (e != cudaSuccess) return e;
            if (K > 1)
                k_commit_conv<__nv_bfloat16><<<counted(dim3(Lg, B)), 256, 0, st>>>(
                    B, N, A, C, K, cap, Pcap, cvec, static_cast<const __nv_bfloat16*>(x),
                    static_cast<__nv_bfloat16*>(conv_state), acc_nodes, acc_len, prefix_len, pg);
        } else {
            e = commit_gdn_dims<float>(dk, dv, B, N, A, Lg, Hk, Hv, K, cap, Pcap, x, conv_w, conv_state, beta, decay,
                                       S, acc_nodes, acc_len, prefix_len, pg, st);
            if (e != cudaSuccess) return e;
            if (K > 1)
                k_commit_conv<float><<<counted(dim3(Lg, B)), 256, 0, st>>>(B, N, A, C, K, cap, Pcap, cvec, static_cast<const float*>(x),
                                                                  static_cast<float*>(conv_state), acc_nodes, acc_len,
                                                                  prefix_len, pg);
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    k_commit_final<<<counted((B + 127) / 128), 128, 0, st>>>(B, N, A, cap, Pcap, acc_nodes, acc_len, prefix_len, src_row,
                                                    dst_pos, status, pg);
    return cudaGetLastError();
}

}  // namespace ddt
