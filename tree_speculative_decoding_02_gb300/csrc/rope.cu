// rope.cu -- ddt_rope_tree: rotary position embedding of the tree rows at their own
// positions, prefix_len + depth.
//
// "DDTree on vLLM: candid research notes", section "Where the next step is": position
// and RoPE correctness by branch depth is one of the blockers.  Nodes of one depth share
// a position ("From Tree-Based Speculative Decoding to Drafter Training", section "The
// Architecture of DDTree"), so siblings get the same rotation and a node's rotation
// follows from its depth, not its row.
//
// One CTA per (node, request): the cos/sin of the node's position are formed once in
// shared memory (angles in fp64 and reduced to [-pi, pi] before the fp32 sin/cos, since
// position * frequency reaches 3e4 radians and more), then every (layer, head) row of q and
// of the tree keys of that node is rotated in place.  Rotation pairs (i, i + rot/2) of the
// first rot_dim channels, frequency theta^(-2i/rot_dim); channels past rot_dim are kept.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace ddt {

template <typename T>
__global__ void __launch_bounds__(256) k_rope_tree(int L, int B, int N, int Hq, int Hkv, int d, int rot, double theta,
                                                   const int32_t* __restrict__ position,
                                                   const int32_t* __restrict__ n_nodes, T* __restrict__ q,
                                                   T* __restrict__ k) {
    extern __shared__ float cs[];  // [rot/2] cos, then [rot/2] sin
    const int n = blockIdx.x, b = blockIdx.y;
    const int half = rot / 2;
    const int nn = n_nodes[b];
    if (n >= nn || nn > N) return;  // padding rows are left as they are
    const double pos = (double)position[(long)b * N + n];
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        const double inv = pow(theta, -2.0 * i / (double)rot);
        const double a = remainder(pos * inv, 2.0 * M_PI);
        float s, c;
        sincosf((float)a, &s, &c);
        cs[i] = c;
        cs[half + i] = s;
    }
    __syncthreads();
    const int nq = q ? Hq : 0;  // q may be absent: keys only
    const int rows = L * (nq + Hkv);
    for (int e = threadIdx.x; e < rows * half; e += blockDim.x) {
        const int rw = e / half, i = e % half;
        const int l = rw / (nq + Hkv), hh = rw % (nq + Hkv);
        T* row = hh < nq ? q + ((((long)l * B + b) * N + n) * Hq + hh) * d
                         : k + ((((long)l * B + b) * N + n) * Hkv + (hh - nq)) * d;
        const float x0 = to_f32(row[i]), x1 = to_f32(row[i + half]);
        const float c = cs[i], s = cs[half + i];
        // one fused multiply-add each, spelled out (the attention kernel's q staging does
        // the same operations, so a rotation there equals a rotation here bit for bit)
        row[i] = from_f32<T>(__fmaf_rn(x0, c, __fmul_rn(-x1, s)));
        row[i + half] = from_f32<T>(__fmaf_rn(x1, c, __fmul_rn(x0, s)));
    }
}

cudaError_t launch_rope_tree(int L, int B, int N, int Hq, int Hkv, int d, int rot, double theta, ddt_dtype dtype,
                             const int32_t* position, const int32_t* n_nodes, void* q, void* k, cudaStream_t st) {
    const size_t smem = sizeof(float) * rot;
    dim3 grid(N, B);
    if (dtype == DDT_BF16)
        k_rope_tree<__nv_bfloat16><<<counted(grid), 256, smem, st>>>(L, B, N, Hq, Hkv, d, rot, theta, position,
                                                                     n_nodes, static_cast<__nv_bfloat16*>(q),
                                                                     static_cast<__nv_bfloat16*>(k));
    else
        k_rope_tree<float><<<counted(grid), 256, smem, st>>>(L, B, N, Hq, Hkv, d, rot, theta, position, n_nodes,
                                                             static_cast<float*>(q), static_cast<float*>(k));
    return cudaGetLastError();
}

// The cos/sin table of every tree row's position (the same angles, formed the same way,
// as k_rope_tree): table [B][N][rot] floats, cos in [0, rot/2), sin in [rot/2, rot).  The
// attention kernels read it to rotate q while staging it (rows of padding nodes are left
// unset: their q rows are never read).
__global__ void __launch_bounds__(128) k_rope_table(int N, int rot, double theta, const int32_t* __restrict__ position,
                                                    const int32_t* __restrict__ n_nodes, float* __restrict__ table) {
    const int n = blockIdx.x, b = blockIdx.y;
    const int half = rot / 2;
    const int nn = n_nodes[b];
    if (n >= nn || nn > N) return;
    const double pos = (double)position[(long)b * N + n];
    float* t = table + ((long)b * N + n) * rot;
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        const double inv = pow(theta, -2.0 * i / (double)rot);
        const double a = remainder(pos * inv, 2.0 * M_PI);
        float s, c;
        sincosf((float)a, &s, &c);
        t[i] = c;
        t[half + i] = s;
    }
}

cudaError_t launch_rope_table(int B, int N, int rot, double theta, const int32_t* position, const int32_t* n_nodes,
                              float* table, cudaStream_t st) {
    k_rope_table<<<counted(dim3(N, B)), 128, 0, st>>>(N, rot, theta, position, n_nodes, table);
    return cudaGetLastError();
}

}  // namespace ddt
