// common.cuh -- small device helpers shared by the kernels of the DDTree round library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ddt.h"

namespace ddt {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;

// ------------------------------------------------------------------ element loads
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Load 8 consecutive elements (16 B for bf16, 32 B for fp32) as floats.  `p` must be
// aligned to the vector width.
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    float4 a = __ldg(reinterpret_cast<const float4*>(p));
    float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Streaming (read-once) variants: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ void load8_stream(const __nv_bfloat16* p, float (&v)[8]) {
    uint4 u = ld_stream_u4(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void load8_stream(const float* p, float (&v)[8]) {
    uint4 a = ld_stream_u4(p);
    uint4 b = ld_stream_u4(reinterpret_cast<const uint4*>(p) + 1);
    v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
    v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
    v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
    v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
}

__device__ __forceinline__ bool finite_f32(float v) {
    return (__float_as_uint(v) & 0x7f800000u) != 0x7f800000u;
}

// ----------------------------------------------------------- ranked (value, id) keys
// Order used for top-k and argmax: larger value first, then smaller id.  Empty
// entries carry id = INT32_MAX and value = -inf so they lose to every real entry.
struct VId {
    float v;
    int id;
};
__device__ __forceinline__ bool beats(float av, int aid, float bv, int bid) {
    return av > bv || (av == bv && aid < bid);
}
__device__ __forceinline__ VId vid_empty() { return VId{-__int_as_float(0x7f800000), 0x7fffffff}; }

// Warp-distributed sorted list of the best `k` (k <= 32) entries: lane r holds the
// entry of rank r; lanes >= k hold the empty entry.  insert() offers one candidate per
// lane; entries that beat the current k-th best are inserted one at a time.
struct WarpTopK {
    float v;
    int id;
    int k;
    __device__ __forceinline__ void init(int k_) {
        k = k_;
        VId e = vid_empty();
        v = e.v;
        id = e.id;
    }
    __device__ __forceinline__ void insert(float cv, int cid) {
        const int lane = threadIdx.x & 31;
        float tv = __shfl_sync(kFull, v, k - 1);
        int tid = __shfl_sync(kFull, id, k - 1);
        unsigned mask = __ballot_sync(kFull, beats(cv, cid, tv, tid));
        while (mask) {
            const int src = __ffs(mask) - 1;
            const float xv = __shfl_sync(kFull, cv, src);
            const int xid = __shfl_sync(kFull, cid, src);
            // rank of x = number of entries that beat it
            const unsigned better = __ballot_sync(kFull, beats(v, id, xv, xid));
            const int pos = __popc(better);
            const float upv = __shfl_up_sync(kFull, v, 1);
            const int upid = __shfl_up_sync(kFull, id, 1);
            if (lane == pos) {
                v = xv;
                id = xid;
            } else if (lane > pos && lane < k) {
                v = upv;
                id = upid;
            }
            mask &= ~(1u << src);
            tv = __shfl_sync(kFull, v, k - 1);
            tid = __shfl_sync(kFull, id, k - 1);
            mask &= __ballot_sync(kFull, beats(cv, cid, tv, tid));
        }
    }
};

// Bitonic networks over one (value, id) entry per lane, best first in the beats order.
// cmpx: exchange with lane ^ stride and keep the better (or the worse) of the pair.
__device__ __forceinline__ void cmpx(float& v, int& id, int stride, bool keep_better) {
    const float ov = __shfl_xor_sync(kFull, v, stride);
    const int oid = __shfl_xor_sync(kFull, id, stride);
    if (beats(ov, oid, v, id) == keep_better) {
        v = ov;
        id = oid;
    }
}
// sorts the warp's 32 entries, best in lane 0
__device__ __forceinline__ void warp_sort_best_first(float& v, int& id) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1)
            cmpx(v, id, stride, ((lane & stride) == 0) == ((lane & size) == 0));
}
// (v, id) and (bv, bid) each sorted best first across the warp: leaves the best 32 of
// their union in (v, id), sorted (the lane-wise better of one list and the other one
// reversed is bitonic and holds the best 32; a half-cleaner cascade sorts it)
__device__ __forceinline__ void warp_merge_best_first(float& v, int& id, float bv, int bid) {
    const int lane = threadIdx.x & 31;
    const float rv = __shfl_sync(kFull, bv, 31 - lane);
    const int rid = __shfl_sync(kFull, bid, 31 - lane);
    if (beats(rv, rid, v, id)) {
        v = rv;
        id = rid;
    }
#pragma unroll
    for (int stride = 16; stride > 0; stride >>= 1) cmpx(v, id, stride, (lane & stride) == 0);
}

// ------------------------------------------------------------------ reductions
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
__device__ __forceinline__ int warp_or(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(kFull, v, o);
    return v;
}

}  // namespace ddt
