// gdn.cu -- ddt_tree_gdn: branch-local gated delta rule with short conv over a tree.
//
// "DDTree on vLLM: candid research notes", sections "Why hybrid attention makes it hard"
// and "Where the next step is": each node reads the GDN and conv state of its parent and
// writes scratch, never the committed state.  The rule itself is the gated delta rule
// of Yang, Kautz and Hatamizadeh, "Gated Delta Networks" (ICLR 2025).
//
// No per-node state is ever materialised.  Along a root-to-node path the recurrence
//   S_t = a_t S_p + u_t k_t^T,   u_t = b_t (v_t - a_t S_p k_t)
// unrolls (the chunked "WY" form of Yang et al., "Parallelizing Linear Transformers with
// the Delta Rule over Sequence Length", NeurIPS 2024) to
//   S_t = g_t S0 + sum_{s in anc(t)+t} G_ts u_s k_s^T,       g_t = prod_{path} a,
//   u_t = b_t (v_t - g_t S0 k_t) - sum_{s in anc(t)} b_t G_ts (k_s . k_t) u_s,
//   o_t = g_t S0 q_t + sum_{s in anc(t)+t} G_ts (k_s . q_t) u_s,
// with G_ts the product of the decays strictly below s down to t.  Every sum runs over
// the node's own ancestors only, which is exactly the branch-local semantics: siblings
// never meet.  The dense part is S0 k_t and S0 q_t for all nodes; the rest is sparse
// along ancestor chains.  One CTA owns one (layer, request, value head) and reads S0
// once from HBM.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace ddt {

namespace {
constexpr int kMD = kGdnMaxDepth;
constexpr int kNT = 16;  // nodes per thread per dense pass
}  // namespace

size_t gdn_smem_bytes(int N, int dk, int dv) {
    size_t b = 0;
    b += sizeof(float) * (size_t)N * (dk + 4) * 2;  // qh, kh
    b += sizeof(float) * (size_t)N * dv * 2;        // vv (-> R -> u), oq
    b += sizeof(int) * (size_t)N * kMD;             // ancestor lists
    b += sizeof(float) * (size_t)N * kMD * 2;       // coefA, coefB
    b += sizeof(float) * (size_t)N * 4;             // bself, gcum, beta, decay
    b += sizeof(int) * (size_t)N * 2;               // depth, parent
    return (b + 15) & ~(size_t)15;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.f + __expf(-z)); }

template <typename Tin, typename Tout, int DK, int DV>
__global__ void __launch_bounds__(256) k_gdn_tree(int B, int N, int Hk, int Hv, int K, const Tin* __restrict__ x,
                                                   const Tin* __restrict__ conv_w,
                                                   const Tin* __restrict__ conv_state,
                                                   const float* __restrict__ beta, const float* __restrict__ decay,
                                                   const float* __restrict__ S, const int32_t* __restrict__ parent,
                                                   const int32_t* __restrict__ n_nodes, Tout* __restrict__ o,
                                                   int32_t* __restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int h = blockIdx.x, b = blockIdx.y, l = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int C = 2 * Hk * DK + Hv * DV;
    const int g = h / (Hv / Hk);
    const long lb = (long)l * B + b;

    float* qh = reinterpret_cast<float*>(smem_raw);          // [N][DK+4]
    float* kh = qh + (size_t)N * (DK + 4);                   // [N][DK+4]
    float* vv = kh + (size_t)N * (DK + 4);                   // [N][DV]
    float* oq = vv + (size_t)N * DV;                         // [N][DV]
    float* cA = oq + (size_t)N * DV;                         // [N][kMD]
    float* cB = cA + (size_t)N * kMD;                        // [N][kMD]
    float* bself = cB + (size_t)N * kMD;                     // [N]
    float* gcum = bself + N;                                 // [N]
    float* sbeta = gcum + N;                                 // [N]
    float* sdec = sbeta + N;                                 // [N]
    int* alist = reinterpret_cast<int*>(sdec + N);           // [N][kMD]
    int* sdep = alist + (size_t)N * kMD;                     // [N]
    int* spar = sdep + N;                                    // [N]
    __shared__ int s_err;

    const int nn = n_nodes[b];
    if (tid == 0) s_err = (nn < 1 || nn > N) ? DDT_ERR_TREE : DDT_OK;
    __syncthreads();
    const int nv = (s_err == DDT_OK) ? nn : 0;
    // ---- phase 0: tree check, ancestor lists, gates
    for (int n = tid; n < nv; n += 256) {
        const int p = parent[(long)b * N + n];
        spar[n] = p;
        if ((n == 0 && p != -1) || (n > 0 && (p < 0 || p >= n))) atomicExch(&s_err, DDT_ERR_TREE);
        sbeta[n] = beta[(lb * N + n) * Hv + h];
        sdec[n] = decay[(lb * N + n) * Hv + h];
    }
    __syncthreads();
    if (s_err == DDT_OK) {
        for (int n = tid; n < nn; n += 256) {
            int d = 0;
            for (int a = spar[n]; a >= 0; a = spar[a]) {
                if (d >= kMD) {
                    atomicExch(&s_err, DDT_ERR_UNSUPPORTED);
                    break;
                }
                alist[n * kMD + d++] = a;
            }
            sdep[n] = d;
        }
    }
    __syncthreads();
    if (tid == 0 && h == 0 && l == 0) status[b] = s_err;
    Tout* ob = o + lb * N * Hv * DV;
    if (s_err != DDT_OK) {
        for (int e = tid; e < N * DV; e += 256) ob[((long)(e / DV) * Hv + h) * DV + e % DV] = from_f32<Tout>(0.f);
        return;
    }

    // ---- phase 1: conv + SiLU along each node's ancestor path, L2 norms (warp per node)
    const Tin* xb = x + lb * N * C;
    const Tin* cs = conv_state + lb * (K - 1) * C;
    const Tin* wl = conv_w + (long)l * C * K;
    const float qscale = rsqrtf((float)DK);
    for (int n = warp; n < nn; n += 8) {
        const int dep = sdep[n];
        int chain[8];  // rows 0..K-1 steps up the path (K <= 8)
        chain[0] = n;
#pragma unroll
        for (int j = 1; j < 8; ++j) chain[j] = (j <= dep) ? alist[n * kMD + j - 1] : -1;
        auto conv = [&](int c) -> float {
            float acc = 0.f;
            for (int j = 0; j < K; ++j) {
                const int back = K - 1 - j;
                const float in = (back <= dep) ? to_f32(xb[(long)chain[back] * C + c])
                                               : to_f32(cs[(long)(K - 1 - (back - dep)) * C + c]);
                acc = fmaf(to_f32(wl[(long)c * K + j]), in, acc);
            }
            return silu_f(acc);
        };
        float yq[DK / 32], yk[DK / 32];
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int e = 0; e < DK / 32; ++e) {
            yq[e] = conv(g * DK + lane + 32 * e);
            yk[e] = conv(Hk * DK + g * DK + lane + 32 * e);
            sq = fmaf(yq[e], yq[e], sq);
            sk = fmaf(yk[e], yk[e], sk);
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        const float rq = rsqrtf(sq + 1e-6f) * qscale, rk = rsqrtf(sk + 1e-6f);
#pragma unroll
        for (int e = 0; e < DK / 32; ++e) {
            qh[n * (DK + 4) + lane + 32 * e] = yq[e] * rq;
            kh[n * (DK + 4) + lane + 32 * e] = yk[e] * rk;
        }
#pragma unroll
        for (int e = 0; e < DV / 32; ++e) vv[n * DV + lane + 32 * e] = conv(2 * Hk * DK + h * DV + lane + 32 * e);
    }
    __syncthreads();

    // ---- phase 2: sparse coefficients along each ancestor chain (warp per node)
    for (int t = warp; t < nn; t += 8) {
        const int dep = sdep[t];
        float dq = 0.f;
#pragma unroll
        for (int e = 0; e < DK / 32; ++e) dq = fmaf(qh[t * (DK + 4) + lane + 32 * e], kh[t * (DK + 4) + lane + 32 * e], dq);
        dq = warp_sum(dq);
        float gam = sdec[t];
        const float bt = sbeta[t];
        for (int m = 0; m < dep; ++m) {
            const int s = alist[t * kMD + m];
            float dk_ = 0.f, dq_ = 0.f;
#pragma unroll
            for (int e = 0; e < DK / 32; ++e) {
                const float ks = kh[s * (DK + 4) + lane + 32 * e];
                dk_ = fmaf(kh[t * (DK + 4) + lane + 32 * e], ks, dk_);
                dq_ = fmaf(qh[t * (DK + 4) + lane + 32 * e], ks, dq_);
            }
            dk_ = warp_sum(dk_);
            dq_ = warp_sum(dq_);
            if (lane == 0) {
                cA[t * kMD + m] = bt * gam * dk_;
                cB[t * kMD + m] = gam * dq_;
            }
            gam *= sdec[s];
        }
        if (lane == 0) {
            bself[t] = dq;
            gcum[t] = gam;
        }
    }
    __syncthreads();

    // ---- phase 3: dense S0 k_t and S0 q_t, fused into R_t and g_t S0 q_t
    {
        constexpr int kHalves = 256 / DV;
        const int jj = tid % DV, half = tid / DV;
        const float* Srow = S + ((lb * Hv + h) * DV + jj) * (long)DK;
        for (int tb = 0; tb < nn; tb += kHalves * kNT) {
            const int t0 = tb + half * kNT;
            float ak[kNT], aq[kNT];
#pragma unroll
            for (int u = 0; u < kNT; ++u) ak[u] = aq[u] = 0.f;
            if (t0 < nn) {
                for (int i = 0; i < DK; i += 4) {
                    const float4 s4 = __ldg(reinterpret_cast<const float4*>(Srow + i));
#pragma unroll
                    for (int u = 0; u < kNT; ++u) {
                        const int t = min(t0 + u, nn - 1);
                        const float4 k4 = *reinterpret_cast<const float4*>(kh + t * (DK + 4) + i);
                        const float4 q4 = *reinterpret_cast<const float4*>(qh + t * (DK + 4) + i);
                        ak[u] = fmaf(s4.x, k4.x, fmaf(s4.y, k4.y, fmaf(s4.z, k4.z, fmaf(s4.w, k4.w, ak[u]))));
                        aq[u] = fmaf(s4.x, q4.x, fmaf(s4.y, q4.y, fmaf(s4.z, q4.z, fmaf(s4.w, q4.w, aq[u]))));
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kNT; ++u) {
                const int t = t0 + u;
                if (t < nn) {
                    vv[t * DV + jj] = sbeta[t] * (vv[t * DV + jj] - gcum[t] * ak[u]);
                    oq[t * DV + jj] = gcum[t] * aq[u];
                }
            }
        }
    }
    __syncthreads();

    // ---- phase 4: per value channel, forward substitution down the tree and outputs
    if (tid < DV) {
        const int jj = tid;
        for (int t = 0; t < nn; ++t) {
            const int dep = sdep[t];
            float u = vv[t * DV + jj];
            float ot = oq[t * DV + jj];
            for (int m = 0; m < dep; ++m) {
                const float us = vv[alist[t * kMD + m] * DV + jj];
                u = fmaf(-cA[t * kMD + m], us, u);
                ot = fmaf(cB[t * kMD + m], us, ot);
            }
            ot = fmaf(bself[t], u, ot);
            vv[t * DV + jj] = u;
            ob[((long)t * Hv + h) * DV + jj] = from_f32<Tout>(ot);
        }
    }
    for (int e = nn * DV + tid; e < N * DV; e += 256) ob[((long)(e / DV) * Hv + h) * DV + e % DV] = from_f32<Tout>(0.f);
}

template <typename Tin, typename Tout, int DK, int DV>
static cudaError_t gdn_go(int L, int B, int N, int Hk, int Hv, int K, const void* x, const void* w, const void* cs,
                          const float* beta, const float* decay, const float* S, const int32_t* parent,
                          const int32_t* nn, void* o, int32_t* status, cudaStream_t st) {
    const size_t smem = gdn_smem_bytes(N, DK, DV);
    cudaError_t e =
        cudaFuncSetAttribute(k_gdn_tree<Tin, Tout, DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(Hv, B, L);
    k_gdn_tree<Tin, Tout, DK, DV><<<counted(grid), 256, smem, st>>>(
        B, N, Hk, Hv, K, static_cast<const Tin*>(x), static_cast<const Tin*>(w), static_cast<const Tin*>(cs), beta,
        decay, S, parent, nn, static_cast<Tout*>(o), status);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
static cudaError_t gdn_dims(int L, int B, int N, int Hk, int Hv, int dk, int dv, int K, const void* x, const void* w,
                            const void* cs, const float* beta, const float* decay, const float* S,
                            const int32_t* parent, const int32_t* nn, void* o, int32_t* status, cudaStream_t st) {
#define DDT_GDN_CASE(A, Bv)                                                                                      \
    if (dk == A && dv == Bv)                                                                                     \
        return gdn_go<Tin, Tout, A, Bv>(L, B, N, Hk, Hv, K, x, w, cs, beta, decay, S, parent, nn, o, status, st);
    DDT_GDN_CASE(32, 32)
    DDT_GDN_CASE(64, 64)
    DDT_GDN_CASE(128, 128)
    DDT_GDN_CASE(64, 128)
    DDT_GDN_CASE(128, 64)
#undef DDT_GDN_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_gdn_tree(int L, int B, int N, int Hk, int Hv, int dk, int dv, int K, ddt_dtype in,
                            ddt_dtype out, const void* x, const void* conv_w, const void* conv_state,
                            const float* beta, const float* decay, const float* S, const int32_t* parent,
                            const int32_t* n_nodes, void* o, int32_t* status, cudaStream_t st) {
    if (in == DDT_BF16 && out == DDT_BF16)
        return gdn_dims<__nv_bfloat16, __nv_bfloat16>(L, B, N, Hk, Hv, dk, dv, K, x, conv_w, conv_state, beta, decay,
                                                      S, parent, n_nodes, o, status, st);
    if (in == DDT_BF16 && out == DDT_F32)
        return gdn_dims<__nv_bfloat16, float>(L, B, N, Hk, Hv, dk, dv, K, x, conv_w, conv_state, beta, decay, S,
                                              parent, n_nodes, o, status, st);
    if (in == DDT_F32 && out == DDT_BF16)
        return gdn_dims<float, __nv_bfloat16>(L, B, N, Hk, Hv, dk, dv, K, x, conv_w, conv_state, beta, decay, S,
                                              parent, n_nodes, o, status, st);
    return gdn_dims<float, float>(L, B, N, Hk, Hv, dk, dv, K, x, conv_w, conv_state, beta, decay, S, parent, n_nodes,
                                  o, status, st);
}

// ---------------------------------------------------------------------------------
// Debugging aid: every node's branch-local state S_n formed the literal way the pages
// describe ("DDTree on vLLM", "Why hybrid attention makes it hard": a node reads its
// parent's recurrent state and writes its own scratch copy, never the committed one).
// One CTA per (value head, request, layer) walks the nodes in row order (every parent
// row precedes its children); thread j owns value row j of every state, so a child
// reads back exactly the row its own thread wrote for the parent.  S_node is
// [L][B][N][Hv][dv][dk]; rows of padding nodes (and of a malformed tree) are zeros.
template <typename Tin>
__global__ void __launch_bounds__(128) k_gdn_states(int B, int N, int Hk, int Hv, int dk, int dv, int K,
                                                    const Tin* __restrict__ x, const Tin* __restrict__ conv_w,
                                                    const Tin* __restrict__ conv_state,
                                                    const float* __restrict__ beta, const float* __restrict__ decay,
                                                    const float* __restrict__ S, const int32_t* __restrict__ parent,
                                                    const int32_t* __restrict__ n_nodes, float* __restrict__ S_node) {
    __shared__ float sk[128], sv[128], rnorm;
    __shared__ int bad;
    const int h = blockIdx.x, b = blockIdx.y, l = blockIdx.z, tid = threadIdx.x;
    const int C = 2 * Hk * dk + Hv * dv, g = h / (Hv / Hk);
    const long lb = (long)l * B + b;
    const int nn = n_nodes[b];
    if (tid == 0) {
        int e = nn < 1 || nn > N;
        for (int n = 0; n < nn && !e; ++n) {
            const int p = parent[(long)b * N + n];
            e = (n == 0) ? p != -1 : (p < 0 || p >= n);
        }
        bad = e;
    }
    __syncthreads();
    const size_t mat = (size_t)dv * dk;
    float* out_b = S_node + (size_t)lb * N * Hv * mat;
    const int nv = bad ? 0 : nn;
    const Tin* xb = x + lb * N * C;
    const Tin* cs = conv_state + lb * (K - 1) * C;
    const Tin* wl = conv_w + (long)l * C * K;
    for (int n = 0; n < nv; ++n) {
        // conv window of node n: its own ancestor path, newest last; taps past the root
        // read the committed conv state (row K-2 newest)
        int chain[8], dep = 0;
        chain[0] = n;
        for (int j = 1; j < K; ++j) {
            const int pj = chain[j - 1] >= 0 ? parent[(long)b * N + chain[j - 1]] : -1;
            chain[j] = pj;
            if (pj >= 0) dep = j;
        }
        // the state update needs k (key head g) and v (value head h); q only enters o
        for (int c = tid; c < dk + dv; c += 128) {
            const int ch = c < dk ? Hk * dk + g * dk + c : 2 * Hk * dk + h * dv + (c - dk);
            float acc = 0.f;
            for (int j = 0; j < K; ++j) {
                const int back = K - 1 - j;
                const float in = back <= dep ? to_f32(xb[(long)chain[back] * C + ch])
                                             : to_f32(cs[(long)(K - 1 - (back - dep)) * C + ch]);
                acc = fmaf(to_f32(wl[(long)ch * K + j]), in, acc);
            }
            const float y = acc / (1.f + expf(-acc));  // SiLU
            if (c < dk) sk[c] = y; else sv[c - dk] = y;
        }
        __syncthreads();
        if (tid < 32) {  // k is L2-normalised per key head
            float a = 0.f;
            for (int i = tid; i < dk; i += 32) a = fmaf(sk[i], sk[i], a);
            a = warp_sum(a);
            if (tid == 0) rnorm = 1.f / sqrtf(a + 1e-6f);
        }
        __syncthreads();
        const float rk = rnorm;
        const float al = decay[(lb * N + n) * Hv + h], be = beta[(lb * N + n) * Hv + h];
        const int p = parent[(long)b * N + n];
        for (int j = tid; j < dv; j += 128) {
            const float* Sp = p < 0 ? S + ((size_t)lb * Hv + h) * mat + (size_t)j * dk
                                    : out_b + ((size_t)p * Hv + h) * mat + (size_t)j * dk;
            float* Sn = out_b + ((size_t)n * Hv + h) * mat + (size_t)j * dk;
            float pk = 0.f;
            for (int i = 0; i < dk; ++i) pk = fmaf(Sp[i], sk[i] * rk, pk);
            const float u = be * (sv[j] - al * pk);
            for (int i = 0; i < dk; ++i) Sn[i] = fmaf(al, Sp[i], u * sk[i] * rk);
        }
        __syncthreads();
    }
    for (int n = nv; n < N; ++n)
        for (size_t e = tid; e < mat; e += 128) out_b[((size_t)n * Hv + h) * mat + e] = 0.f;
}

cudaError_t launch_gdn_states(int L, int B, int N, int Hk, int Hv, int dk, int dv, int K, ddt_dtype in,
                              const void* x, const void* conv_w, const void* conv_state, const float* beta,
                              const float* decay, const float* S, const int32_t* parent, const int32_t* n_nodes,
                              float* S_node, cudaStream_t st) {
    if (dk > 128 || dv > 128 || K > 8) return cudaErrorInvalidValue;
    dim3 grid(Hv, B, L);
    if (in == DDT_BF16)
        k_gdn_states<__nv_bfloat16><<<counted(grid), 128, 0, st>>>(
            B, N, Hk, Hv, dk, dv, K, static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(conv_w),
            static_cast<const __nv_bfloat16*>(conv_state), beta, decay, S, parent, n_nodes, S_node);
    else
        k_gdn_states<float><<<counted(grid), 128, 0, st>>>(B, N, Hk, Hv, dk, dv, K, static_cast<const float*>(x),
                                                          static_cast<const float*>(conv_w),
                                                          static_cast<const float*>(conv_state), beta, decay, S,
                                                          parent, n_nodes, S_node);
    return cudaGetLastError();
}

}  // namespace ddt
