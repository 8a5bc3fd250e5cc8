// lowrank.cu -- kvfix_lowrank_apply: out = x + A B per (chunk, layer, KV head).
//
// Method: KVCMAS Eq. 4 (corrected cache = reference + estimated delta), Eq. 7 (a delta
// kept as factors A [rows x r] and B [r x D]), Eq. 8 with a single anchor of weight 1.
//
// Tensor-core path (warp-level bf16 MMA, m16n8k16, float accumulation).  Each warp
// owns 16 token rows of one head: it stages the rows of x through shared memory with
// coalesced 16-byte loads, multiplies its 16 x r slice of A by B (held transposed in
// shared memory) and adds the product to x in float before one rounding to bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace kvfix {

constexpr int kLrWarps = 8;
constexpr int kLrRowsPerWarp = 16;
constexpr int kLrTilesPerCta = 8;  // 16-row tiles per warp per CTA

__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, const uint32_t* b) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// grid = (ceil(n / rows_per_cta), H, C*L).  Row stride in shared memory is D + 8
// elements (D=128: 272 bytes) so that fragment reads are free of bank conflicts.
template <int D>
__global__ void __launch_bounds__(kLrWarps * 32)
lowrank_mma_kernel(const uint16_t* x, Plane p, const uint16_t* __restrict__ A,
                   const uint16_t* __restrict__ B, int rank, uint16_t* out, Plane op) {
    constexpr int kPitch = D + 8;            // bf16 elements per staged row
    constexpr int kNT = D / 8;               // n-tiles of 8 dims
    constexpr int kV = D / 8;                // 16-byte vectors per row
    extern __shared__ __align__(16) uint16_t sm[];
    uint16_t* bt = sm;                                   // [D][rank + 8] (B transposed)
    const int bpitch = rank + 8;
    uint16_t* xs_all = sm + D * bpitch;                  // [warps][16][kPitch]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int h = blockIdx.y;
    const int cl = blockIdx.z;
    const int c = cl / p.layers, l = cl % p.layers;
    const int n = p.tokens;
    const long long unit = (long long)cl * p.heads + h;
    const uint16_t* Au = A + unit * (long long)n * rank;
    const uint16_t* Bu = B + unit * (long long)rank * D;

    for (int i = threadIdx.x; i < rank * D; i += blockDim.x) {
        int k = i / D, e = i % D;
        bt[e * bpitch + k] = Bu[i];
    }
    __syncthreads();

    uint16_t* xs = xs_all + warp * kLrRowsPerWarp * kPitch;
    const int row_base = blockIdx.x * (kLrWarps * kLrRowsPerWarp * kLrTilesPerCta);
    for (int tile = 0; tile < kLrTilesPerCta; ++tile) {
        const int r0 = row_base + (tile * kLrWarps + warp) * kLrRowsPerWarp;
        if (r0 >= n) break;
        const int rows = min(kLrRowsPerWarp, n - r0);
        // stage x rows (coalesced 16-byte vectors)
        for (int i = lane; i < kLrRowsPerWarp * kV; i += 32) {
            int rr = i / kV, v = i % kV;
            uint4 val = make_uint4(0, 0, 0, 0);
            if (rr < rows)
                val = ld_stream(reinterpret_cast<const uint4*>(x + p.row(c, l, r0 + rr) + (long long)h * D + 8 * v));
            *reinterpret_cast<uint4*>(xs + rr * kPitch + 8 * v) = val;
        }
        float acc[kNT][4];
#pragma unroll
        for (int t = 0; t < kNT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
        for (int k0 = 0; k0 < rank; k0 += 16) {
            uint32_t a[4];
            const int ra = r0 + g, rb = r0 + g + 8;
            a[0] = ra < n ? *reinterpret_cast<const uint32_t*>(Au + (long long)ra * rank + k0 + 2 * q) : 0u;
            a[1] = rb < n ? *reinterpret_cast<const uint32_t*>(Au + (long long)rb * rank + k0 + 2 * q) : 0u;
            a[2] = ra < n ? *reinterpret_cast<const uint32_t*>(Au + (long long)ra * rank + k0 + 8 + 2 * q) : 0u;
            a[3] = rb < n ? *reinterpret_cast<const uint32_t*>(Au + (long long)rb * rank + k0 + 8 + 2 * q) : 0u;
#pragma unroll
            for (int t = 0; t < kNT; ++t) {
                uint32_t b[2];
                const uint16_t* bcol = bt + (t * 8 + g) * bpitch + k0 + 2 * q;
                b[0] = *reinterpret_cast<const uint32_t*>(bcol);
                b[1] = *reinterpret_cast<const uint32_t*>(bcol + 8);
                mma_bf16_16816(acc[t], a, b);
            }
        }
        __syncwarp();
        // epilogue: x + AB in float, one rounding, written back into the staging rows
#pragma unroll
        for (int t = 0; t < kNT; ++t) {
            const int col = t * 8 + 2 * q;
            __nv_bfloat162* p0 = reinterpret_cast<__nv_bfloat162*>(xs + g * kPitch + col);
            __nv_bfloat162* p1 = reinterpret_cast<__nv_bfloat162*>(xs + (g + 8) * kPitch + col);
            float2 x0 = __bfloat1622float2(*p0);
            float2 x1 = __bfloat1622float2(*p1);
            *p0 = __floats2bfloat162_rn(x0.x + acc[t][0], x0.y + acc[t][1]);
            *p1 = __floats2bfloat162_rn(x1.x + acc[t][2], x1.y + acc[t][3]);
        }
        __syncwarp();
        for (int i = lane; i < rows * kV; i += 32) {
            int rr = i / kV, v = i % kV;
            uint4 val = *reinterpret_cast<const uint4*>(xs + rr * kPitch + 8 * v);
            st_stream(reinterpret_cast<uint4*>(out + op.row(c, l, r0 + rr) + (long long)h * D + 8 * v), val);
        }
        __syncwarp();
    }
}

cudaError_t launch_lowrank(const uint16_t* x, const kvfix_kv_desc& d, const uint16_t* A,
                           const uint16_t* B, int rank, uint16_t* out, const kvfix_kv_desc& od,
                           cudaStream_t s) {
    Plane p = plane_of(d), op = plane_of(od);
    if (p.chunks == 0 || p.layers == 0 || p.tokens == 0) return cudaSuccess;
    const int rows_per_cta = kLrWarps * kLrRowsPerWarp * kLrTilesPerCta;
    dim3 grid((p.tokens + rows_per_cta - 1) / rows_per_cta, p.heads, p.chunks * p.layers);
    const size_t smem = sizeof(uint16_t) * ((size_t)p.dim * (rank + 8) +
                                            (size_t)kLrWarps * kLrRowsPerWarp * (p.dim + 8));
    cudaError_t e;
    if (p.dim == 128) {
        e = cudaFuncSetAttribute(lowrank_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        lowrank_mma_kernel<128><<<grid, kLrWarps * 32, smem, s>>>(x, p, A, B, rank, out, op);
    } else {
        e = cudaFuncSetAttribute(lowrank_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        lowrank_mma_kernel<64><<<grid, kLrWarps * 32, smem, s>>>(x, p, A, B, rank, out, op);
    }
    return cudaGetLastError();
}

}  // namespace kvfix
