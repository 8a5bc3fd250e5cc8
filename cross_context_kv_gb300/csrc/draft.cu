// draft.cu -- kvfix_draft_rank: rank cached rows by the softmax attention mass of the
// draft queries, keep the best k rows, optionally overwrite them with fresh rows.
//
// Method: Budgeted Cache Repair, section 3 ("The repair": row score a_j summed over
// layers after the first, steps and heads of softmax(Q K~^T / sqrt(d_head))), App. B
// Algorithm 2 (grouped-query keys expanded to query heads) and Algorithm 1 step 6
// (the selected rows' K and V are overwritten before use); KVCMAS Eq. 3.
//
// Pipeline (one unit = chunk, layer >= layer_begin, KV head; its G = steps x
// q_heads/kv_heads <= 16 query rows share the unit's keys):
//   1. logits:  tensor-core QK^T per 128-key tile -> logits in the workspace, plus the
//               tile's per-query (max, sum exp) partials;
//   2. stats:   per (unit, query) combine the tile partials into (max, sum exp);
//   3. accum:   per key, sum over units (layer-major, then head) and queries of
//               exp(z - max) / sum, float per unit, double across units;
//   4. select:  top-k of the double scores (ties to the lower index);
//   5. repair:  copy the selected rows of every layer and head from the fresh planes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace kvfix {

static __device__ unsigned int g_status_draft;

unsigned read_status_draft(cudaStream_t stream) {
    unsigned h = 0, zero = 0;
    cudaMemcpyFromSymbolAsync(&h, g_status_draft, sizeof h, 0, cudaMemcpyDeviceToHost, stream);
    cudaMemcpyToSymbolAsync(g_status_draft, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    cudaStreamSynchronize(stream);
    return h;
}

constexpr int kDrWarps = 8;
constexpr int kDrTile = kDrWarps * 16;  // keys per CTA in the logits pass
constexpr int kDrQ = 16;                // query rows per unit (padded)

struct DraftWs {
    float* logits;   // [units][16][n]
    float2* part;    // [units][tiles][16]  (max, sum exp) of a key tile
    float2* stats;   // [units][16]         (max, 1 / sum exp)
};

static DraftWs carve(void* ws, long long units, int n) {
    const long long tiles = (n + kDrTile - 1) / kDrTile;
    char* p = static_cast<char*>(ws);
    DraftWs w;
    w.logits = reinterpret_cast<float*>(p);
    p += ((sizeof(float) * units * kDrQ * n + 255) / 256) * 256;
    w.part = reinterpret_cast<float2*>(p);
    p += ((sizeof(float2) * units * tiles * kDrQ + 255) / 256) * 256;
    w.stats = reinterpret_cast<float2*>(p);
    return w;
}

size_t draft_workspace_bytes(const kvfix_kv_desc& d, int layer_begin) {
    const long long nl = d.layers > layer_begin ? d.layers - layer_begin : 0;
    const long long units = (long long)d.chunks * nl * d.kv_heads;
    const long long n = d.tokens;
    const long long tiles = (n + kDrTile - 1) / kDrTile;
    size_t b = ((sizeof(float) * units * kDrQ * n + 255) / 256) * 256;
    b += ((sizeof(float2) * units * tiles * kDrQ + 255) / 256) * 256;
    b += ((sizeof(float2) * units * kDrQ + 255) / 256) * 256;
    return b;
}

__device__ __forceinline__ void mma_16816(float* d, const uint32_t* a, const uint32_t* b) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// ---- 1. logits: grid = (tiles, units) ------------------------------------------
template <int D>
__global__ void __launch_bounds__(kDrWarps * 32)
draft_logits_kernel(const uint16_t* __restrict__ k, Plane p, const uint16_t* __restrict__ q,
                    int steps, int q_heads, int layer_begin, int G, DraftWs ws) {
    constexpr int kPitch = D + 8;
    constexpr int kV = D / 8;
    __shared__ __align__(16) uint16_t qs[kDrQ * kPitch];
    __shared__ __align__(16) uint16_t ks[kDrWarps][16 * kPitch];
    __shared__ float2 red[kDrWarps][kDrQ];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, qd = lane & 3;
    const int n = p.tokens, H = p.heads;
    const int nl = p.layers - layer_begin;
    const long long unit = blockIdx.y;
    const int kvh = (int)(unit % H);
    const int l = layer_begin + (int)((unit / H) % nl);
    const int c = (int)(unit / ((long long)H * nl));
    const int group = q_heads / H;
    // queries of this unit: row i = t*group + m  <->  q[c][l][t][kvh*group + m]
    for (int i = threadIdx.x; i < kDrQ * kV; i += blockDim.x) {
        int row = i / kV, v = i % kV;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (row < G) {
            int t = row / group, m = row % group;
            const uint16_t* src = q + ((((long long)c * p.layers + l) * steps + t) * q_heads + kvh * group + m) * D;
            val = *reinterpret_cast<const uint4*>(src + 8 * v);
        }
        *reinterpret_cast<uint4*>(qs + row * kPitch + 8 * v) = val;
    }
    const int j0 = blockIdx.x * kDrTile + warp * 16;
    uint16_t* kw = ks[warp];
    for (int i = lane; i < 16 * kV; i += 32) {
        int rr = i / kV, v = i % kV;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (j0 + rr < n)
            val = ld_stream(reinterpret_cast<const uint4*>(k + p.row(c, l, j0 + rr) + (long long)kvh * D + 8 * v));
        *reinterpret_cast<uint4*>(kw + rr * kPitch + 8 * v) = val;
    }
    __syncthreads();
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int k0 = 0; k0 < D; k0 += 16) {
        uint32_t a[4];
        a[0] = *reinterpret_cast<const uint32_t*>(kw + g * kPitch + k0 + 2 * qd);
        a[1] = *reinterpret_cast<const uint32_t*>(kw + (g + 8) * kPitch + k0 + 2 * qd);
        a[2] = *reinterpret_cast<const uint32_t*>(kw + g * kPitch + k0 + 8 + 2 * qd);
        a[3] = *reinterpret_cast<const uint32_t*>(kw + (g + 8) * kPitch + k0 + 8 + 2 * qd);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            uint32_t b[2];
            const uint16_t* qrow = qs + (t * 8 + g) * kPitch + k0 + 2 * qd;
            b[0] = *reinterpret_cast<const uint32_t*>(qrow);
            b[1] = *reinterpret_cast<const uint32_t*>(qrow + 8);
            mma_16816(acc[t], a, b);
        }
    }
    const float scale = rsqrtf((float)D);
    // acc[t][0,1]: key j0+g, queries t*8+2qd, +1; acc[t][2,3]: key j0+g+8.
    const int ja = j0 + g, jb = j0 + g + 8;
    float* lg = ws.logits + unit * kDrQ * (long long)n;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int qi = t * 8 + 2 * qd + e;
            float za = acc[t][e] * scale, zb = acc[t][2 + e] * scale;
            if (ja < n) lg[(long long)qi * n + ja] = za;
            if (jb < n) lg[(long long)qi * n + jb] = zb;
            // tile partial: max and sum exp over this warp's 16 keys (lanes sharing qd)
            float m = fmaxf(ja < n ? za : -INFINITY, jb < n ? zb : -INFINITY);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            float s = (ja < n ? expf(za - m) : 0.f) + (jb < n ? expf(zb - m) : 0.f);
            if (m == -INFINITY) s = 0.f;
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (g == 0) red[warp][qi] = make_float2(m, s);
        }
    }
    __syncthreads();
    if (threadIdx.x < kDrQ) {
        const int qi = threadIdx.x;
        float m = -INFINITY;
        for (int w = 0; w < kDrWarps; ++w) m = fmaxf(m, red[w][qi].x);
        float s = 0.f;
        if (m != -INFINITY)
            for (int w = 0; w < kDrWarps; ++w)
                if (red[w][qi].x != -INFINITY) s += red[w][qi].y * expf(red[w][qi].x - m);
        ws.part[(unit * gridDim.x + blockIdx.x) * kDrQ + qi] = make_float2(m, s);
    }
}

// ---- 2. stats: grid = units, 16 threads x ... ------------------------------------
__global__ void draft_stats_kernel(DraftWs ws, int tiles) {
    const long long unit = blockIdx.x;
    const int qi = threadIdx.x;
    if (qi >= kDrQ) return;
    float m = -INFINITY;
    for (int t = 0; t < tiles; ++t) m = fmaxf(m, ws.part[(unit * tiles + t) * kDrQ + qi].x);
    float s = 0.f;
    for (int t = 0; t < tiles; ++t) {
        float2 pt = ws.part[(unit * tiles + t) * kDrQ + qi];
        if (pt.x != -INFINITY) s += pt.y * expf(pt.x - m);
    }
    ws.stats[unit * kDrQ + qi] = make_float2(m, s > 0.f ? 1.0f / s : 0.f);
}

// ---- 3. accumulate: grid = (ceil(n/256), chunks) -----------------------------------
constexpr int kAccThreads = 256;

__global__ void __launch_bounds__(kAccThreads)
draft_accum_kernel(DraftWs ws, int n, long long units_per_chunk, int G, double* scores) {
    __shared__ float2 st[64][kDrQ];
    const int c = blockIdx.y;
    const int j = blockIdx.x * kAccThreads + threadIdx.x;
    double acc = 0.0;
    for (long long u0 = 0; u0 < units_per_chunk; u0 += 64) {
        const int nu = (int)min(64ll, units_per_chunk - u0);
        __syncthreads();
        for (int i = threadIdx.x; i < nu * kDrQ; i += blockDim.x)
            st[i / kDrQ][i % kDrQ] = ws.stats[((long long)c * units_per_chunk + u0 + i / kDrQ) * kDrQ + i % kDrQ];
        __syncthreads();
        if (j < n) {
            for (int uu = 0; uu < nu; ++uu) {
                const long long unit = (long long)c * units_per_chunk + u0 + uu;
                const float* lg = ws.logits + unit * kDrQ * (long long)n + j;
                float f = 0.f;
                for (int qi = 0; qi < G; ++qi) f += expf(lg[(long long)qi * n] - st[uu][qi].x) * st[uu][qi].y;
                acc += (double)f;
            }
        }
    }
    if (j < n) scores[(long long)c * n + j] = acc;
}

// ---- 4. select (double keys) --------------------------------------------------------
constexpr int kSelThreads2 = 1024;
constexpr int kSelSmemKeys2 = 16384;

__device__ __forceinline__ unsigned long long ordered_f64(double f) {
    unsigned long long u = (unsigned long long)__double_as_longlong(f);
    return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

__device__ int block_exclusive_scan2(int x, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    int inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    __syncthreads();
    if (lane == 31) warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int ws = lane < nw ? warp_sums[lane] : 0;
        int wi = ws;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < nw) warp_sums[lane] = wi - ws;
        if (lane == 31) warp_sums[32] = wi;
    }
    __syncthreads();
    int ex = inc - x + warp_sums[warp];
    *total = warp_sums[32];
    __syncthreads();
    return ex;
}

// Radix select of the k largest 64-bit keys (ties to the lower index).
__global__ void __launch_bounds__(kSelThreads2)
select_f64_kernel(const double* __restrict__ scores, int n, int kk, int32_t* idx) {
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ unsigned hist[256];
    __shared__ int warp_sums[33];
    __shared__ unsigned long long s_prefix;
    __shared__ int s_remaining;
    const int words = (n + 31) / 32;
    uint32_t* bits = reinterpret_cast<uint32_t*>(dyn);
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(dyn + ((sizeof(uint32_t) * words + 15) / 16) * 16);
    const bool cached = n <= kSelSmemKeys2;
    const long long c = blockIdx.x;
    const double* sc = scores + c * n;
    int32_t* out = idx + c * kk;
    const int tid = threadIdx.x;
    auto key_at = [&](int i) -> unsigned long long { return cached ? keys[i] : ordered_f64(sc[i]); };
    for (int w = tid; w < words; w += blockDim.x) bits[w] = 0u;
    if (cached)
        for (int i = tid; i < n; i += blockDim.x) keys[i] = ordered_f64(sc[i]);
    if (tid == 0) {
        s_prefix = 0ull;
        s_remaining = kk;
    }
    __syncthreads();
    if (kk <= 0) return;
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0u;
        __syncthreads();
        const unsigned long long prefix = s_prefix;
        const unsigned long long hi_mask = shift == 56 ? 0ull : ~((1ull << (shift + 8)) - 1ull);
        for (int i = tid; i < n; i += blockDim.x) {
            unsigned long long kv = key_at(i);
            if ((kv & hi_mask) == (prefix & hi_mask)) atomicAdd(&hist[(unsigned)(kv >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 32) {
            unsigned cnt[8];
            unsigned lsum = 0;
#pragma unroll
            for (int qq = 0; qq < 8; ++qq) {
                cnt[qq] = hist[255 - 8 * tid - qq];
                lsum += cnt[qq];
            }
            unsigned inc = lsum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                unsigned y = __shfl_up_sync(0xffffffffu, inc, o);
                if (tid >= o) inc += y;
            }
            const unsigned before = inc - lsum;
            const unsigned rem = (unsigned)s_remaining;
            if (before < rem && rem <= inc) {
                unsigned acc = before;
#pragma unroll
                for (int qq = 0; qq < 8; ++qq) {
                    if (acc < rem && rem <= acc + cnt[qq]) {
                        s_prefix = prefix | ((unsigned long long)(255 - 8 * tid - qq) << shift);
                        s_remaining = (int)(rem - acc);
                    }
                    acc += cnt[qq];
                }
            }
        }
        __syncthreads();
    }
    const unsigned long long T = s_prefix;
    const int need_eq = s_remaining;
    const int seg = (n + blockDim.x - 1) / blockDim.x;
    const int i0 = min(n, tid * seg), i1 = min(n, i0 + seg);
    int eq = 0;
    for (int i = i0; i < i1; ++i) eq += (key_at(i) == T);
    int tot;
    int eq_before = block_exclusive_scan2(eq, warp_sums, &tot);
    int cnt = 0;
    for (int i = i0; i < i1; ++i) {
        unsigned long long kv = key_at(i);
        bool take = kv > T;
        if (kv == T) {
            take = eq_before < need_eq;
            ++eq_before;
        }
        if (take) {
            atomicOr(&bits[i >> 5], 1u << (i & 31));
            ++cnt;
        }
    }
    int ob = block_exclusive_scan2(cnt, warp_sums, &tot);
    __syncthreads();
    for (int i = i0; i < i1; ++i)
        if ((bits[i >> 5] >> (i & 31) & 1u) && ob < kk) out[ob++] = i;
}

cudaError_t launch_draft(const uint16_t* k, const kvfix_kv_desc& d, const uint16_t* q, int steps,
                         int q_heads, int layer_begin, int k_rows, int32_t* idx, double* scores,
                         void* ws_ptr, cudaStream_t s) {
    Plane p = plane_of(d);
    const int n = p.tokens;
    const int nl = p.layers - layer_begin;
    const long long units_per_chunk = (long long)nl * p.heads;
    const long long units = units_per_chunk * p.chunks;
    const int G = steps * (q_heads / p.heads);
    cudaError_t e;
    if (p.chunks == 0 || n == 0) return cudaSuccess;
    if (units == 0) {
        e = cudaMemsetAsync(scores, 0, sizeof(double) * (size_t)p.chunks * n, s);
        if (e != cudaSuccess) return e;
    } else {
        DraftWs ws = carve(ws_ptr, units, n);
        const int tiles = (n + kDrTile - 1) / kDrTile;
        if (units > 65535) return cudaErrorInvalidValue;
        dim3 g1(tiles, (unsigned)units);
        if (p.dim == 128)
            draft_logits_kernel<128><<<g1, kDrWarps * 32, 0, s>>>(k, p, q, steps, q_heads, layer_begin, G, ws);
        else
            draft_logits_kernel<64><<<g1, kDrWarps * 32, 0, s>>>(k, p, q, steps, q_heads, layer_begin, G, ws);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        draft_stats_kernel<<<(unsigned)units, 32, 0, s>>>(ws, tiles);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        dim3 g3((n + kAccThreads - 1) / kAccThreads, p.chunks);
        draft_accum_kernel<<<g3, kAccThreads, 0, s>>>(ws, n, units_per_chunk, G, scores);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (k_rows > 0) {
        const int words = (n + 31) / 32;
        size_t smem = ((sizeof(uint32_t) * words + 15) / 16) * 16 + (n <= kSelSmemKeys2 ? sizeof(unsigned long long) * n : 0);
        e = cudaFuncSetAttribute(select_f64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        select_f64_kernel<<<p.chunks, kSelThreads2, smem, s>>>(scores, n, k_rows, idx);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// ---- 5. row repair: grid = (ceil(k/16), L, C) ----------------------------------------
constexpr int kRepThreads = 256;
constexpr int kRepRows = 16;

__global__ void __launch_bounds__(kRepThreads)
row_repair_kernel(uint16_t* io, Plane p, const uint16_t* __restrict__ fresh, Plane fp,
                  const int32_t* __restrict__ idx, int kk) {
    const int l = blockIdx.y, c = blockIdx.z;
    const int row8 = p.heads * p.dim / 8;
    const int i0 = blockIdx.x * kRepRows;
    const int rows = min(kRepRows, kk - i0);
    for (int it = threadIdx.x; it < rows * row8; it += kRepThreads) {
        const int i = i0 + it / row8, v = it % row8;
        const int j = idx[(long long)c * kk + i];
        if (j < 0 || j >= p.tokens) {
            if (v == 0) atomicOr(&g_status_draft, FLAG_BOUNDS);
            continue;
        }
        uint4 val = ld_stream(reinterpret_cast<const uint4*>(fresh + fp.row(c, l, j) + 8ll * v));
        st_stream(reinterpret_cast<uint4*>(io + p.row(c, l, j) + 8ll * v), val);
    }
}

cudaError_t launch_row_repair(uint16_t* io, const kvfix_kv_desc& d, const uint16_t* fresh,
                              const kvfix_kv_desc& fd, const int32_t* idx, int k_rows,
                              cudaStream_t s) {
    Plane p = plane_of(d), fp = plane_of(fd);
    if (k_rows == 0 || p.layers == 0 || p.chunks == 0) return cudaSuccess;
    dim3 grid((k_rows + kRepRows - 1) / kRepRows, p.layers, p.chunks);
    row_repair_kernel<<<grid, kRepThreads, 0, s>>>(io, p, fresh, fp, idx, k_rows);
    return cudaGetLastError();
}

}  // namespace kvfix
