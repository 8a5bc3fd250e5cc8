// common.cuh -- shared device helpers of libkvfix (bf16 vectors, RoPE angles,
// status flags, plane addressing).  Included by every kernel translation unit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace kvfix {

// Device status bits (each translation unit keeps its own word; see internal.h).
enum : unsigned {
    FLAG_BOUNDS = 1u,   // an index in caller data was out of range and skipped
    FLAG_NOSPACE = 2u,  // a payload entry beyond the capacity was skipped
    FLAG_TIMEOUT = 4u,  // a bounded wait gave up
};

// ------------------------------------------------------------- addressing

struct Plane {
    int chunks, layers, tokens, heads, dim;
    long long sc, sl, st;  // element strides of chunk, layer, token
    __host__ __device__ long long row(int c, int l, int t) const {
        return (long long)c * sc + (long long)l * sl + (long long)t * st;
    }
};

inline Plane plane_of(const kvfix_kv_desc& d) {
    Plane p;
    p.chunks = d.chunks;
    p.layers = d.layers;
    p.tokens = d.tokens;
    p.heads = d.kv_heads;
    p.dim = d.head_dim;
    p.sc = d.stride_chunk;
    p.sl = d.stride_layer;
    p.st = d.stride_token;
    return p;
}

// ------------------------------------------------------------- bf16 vectors

// 8 bf16 values = one 16-byte vector.
__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float* f) {
    uint4 v;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return v;
}

// Read-once streaming load / write-once streaming store.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_plain(const uint4* p) {
    return *p;
}

__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// ------------------------------------------------------------- RoPE angles

// Rotation angle delta * theta_i reduced to [-pi, pi] in double, then cos/sin in
// float.  theta_i is computed on the host in double.
__device__ __forceinline__ void rope_cos_sin(int delta, double theta, float* c, float* s) {
    const double kTwoPiHi = 6.283185307179586;       // nearest double to 2 pi
    const double kTwoPiLo = 2.4492935982947064e-16;  // 2 pi - kTwoPiHi
    const double kInvTwoPi = 0.15915494309189535;
    double a = (double)delta * theta;
    double k = rint(a * kInvTwoPi);
    double r = fma(-k, kTwoPiHi, a);
    r = fma(-k, kTwoPiLo, r);
    sincosf((float)r, s, c);
}

// Rotate the pair of 8-wide vectors (x_i, x_{i+D/2}) for i = i0..i0+7.
__device__ __forceinline__ void rotate_pair(float* lo, float* hi, const float* c, const float* s) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        float x0 = lo[k], x1 = hi[k];
        lo[k] = x0 * c[k] - x1 * s[k];
        hi[k] = x1 * c[k] + x0 * s[k];
    }
}

}  // namespace kvfix
