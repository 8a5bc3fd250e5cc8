// common.cuh -- shared device helpers of libkvfix (bf16 vectors, RoPE angles,
// status flags, plane addressing).  Included by every kernel translation unit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "internal.h"

namespace kvfix {

// Device status bits (each translation unit keeps its own word; see internal.h).
enum : unsigned {
    FLAG_BOUNDS = 1u,   // an index in caller data was out of range and skipped
    FLAG_NOSPACE = 2u,  // a payload entry beyond the capacity was skipped
    FLAG_TIMEOUT = 4u,  // a bounded wait gave up
    FLAG_INTERNAL = 8u, // a kernel's own layout check failed; it skipped its work
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

// acc[i] += the 8 bf16 values of v, in order.
__device__ __forceinline__ void add8(const uint4& v, float* acc) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __bfloat1622float2(h[i]);
        acc[2 * i] += t.x;
        acc[2 * i + 1] += t.y;
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
        lo[k] = __fmaf_rn(x0, c[k], __fmul_rn(x1, -s[k]));  // same rounding as the packed form
        hi[k] = __fmaf_rn(x1, c[k], __fmul_rn(x0, s[k]));
    }
}

}  // namespace kvfix

// ------------------------------------------------------------- async bulk copies
// 1-D bulk copies global -> shared completed on an mbarrier (transaction bytes),
// the TMA path for contiguous rows.  Waits are bounded in time: past the limit the
// caller sets a timeout flag instead of spinning on.
namespace kvfix {


__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// One poll; the thread may be suspended (up to kSuspendNs) until the phase completes.
constexpr unsigned kSuspendNs = 1000000;  // 1 ms per poll
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity; false once about kWaitCycles SM
// clocks (~2 s) have passed without completion.
constexpr long long kWaitCycles = 4000000000ll;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

}  // namespace kvfix

namespace kvfix {
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Per-thread asynchronous 16-byte global -> shared copy (bypassing L1); completion is
// counted in the thread's commit groups.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's commit groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
}  // namespace kvfix

// ------------------------------------------------------------- 4-wide (8-byte) helpers
namespace kvfix {
__device__ __forceinline__ void unpack4(const uint2& v, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
    float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
    f[0] = a.x;
    f[1] = a.y;
    f[2] = b.x;
    f[3] = b.y;
}

__device__ __forceinline__ uint2 pack4(const float* f) {
    uint2 v;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
    h[0] = __floats2bfloat162_rn(f[0], f[1]);
    h[1] = __floats2bfloat162_rn(f[2], f[3]);
    return v;
}

__device__ __forceinline__ void add4(const uint2& v, float* acc) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
    float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
    acc[0] += a.x;
    acc[1] += a.y;
    acc[2] += b.x;
    acc[3] += b.y;
}

__device__ __forceinline__ void rotate4(float* lo, float* hi, const float* c, const float* s) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float x0 = lo[k], x1 = hi[k];
        lo[k] = __fmaf_rn(x0, c[k], __fmul_rn(x1, -s[k]));  // same rounding as the packed form
        hi[k] = __fmaf_rn(x1, c[k], __fmul_rn(x0, s[k]));
    }
}

__device__ __forceinline__ void st_stream2(uint2* p, const uint2& v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}
}  // namespace kvfix

// ------------------------------------------------------------- programmatic launch
// Kernels of one call chain (score -> select -> mean correction) are launched with
// programmatic stream serialisation: the next kernel may start once every CTA of the
// previous one has called pdl_trigger(), and must call pdl_wait() before it reads
// anything the previous kernel writes.  Before pdl_wait() a kernel only reads inputs
// that no kernel of the chain writes.  Launched without the attribute (or after a
// kernel that never triggers), pdl_wait() returns at once and order is as usual.
namespace kvfix {
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... Exp, typename... Act>
inline cudaError_t launch_chained(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t s, Act&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Act>(args)...);
}
}  // namespace kvfix
