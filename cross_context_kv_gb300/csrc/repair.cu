// repair.cu -- re-rope, check-layer divergence, top-b probe selection and probe-mean
// correction of reused KV chunks (kvfix_rerope, kvfix_score_topk, kvfix_mean_correct).
//
// Method: AgentKVShift: Correcting Reused KV, "Core idea and method" (steps 1-4 and
// the displayed b, d, w, mu-hat and K_corr equations); KVCMAS section 2.2 / App. A.3
// (re-alignment of cached keys); TokenDance section 4.2 (all agents of a round share
// one rotation pass and one check-layer pass).
//
// Layout: one KV plane is [chunk][layer][token][head][dim] with the heads of a token
// contiguous; rows move as 16-byte vectors of 8 bf16.  A "pair vector" is the two
// 8-wide vectors that rotate-half RoPE mixes: dims [8v, 8v+8) and [8v+D/2, 8v+D/2+8).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace kvfix {

static __device__ unsigned int g_status_repair;

unsigned read_status_repair(cudaStream_t stream) {
    unsigned h = 0, zero = 0;
    cudaMemcpyFromSymbolAsync(&h, g_status_repair, sizeof h, 0, cudaMemcpyDeviceToHost, stream);
    cudaMemcpyToSymbolAsync(g_status_repair, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    cudaStreamSynchronize(stream);
    return h;
}

// Per-CTA table of (cos, sin) of delta*theta_i, i < D/2.
__device__ __forceinline__ void build_table(float2* tab, int delta, const RopeTheta& th, int half,
                                            int tid, int nthreads) {
    for (int i = tid; i < half; i += nthreads) {
        float c, s;
        rope_cos_sin(delta, th.theta[i], &c, &s);
        tab[i] = make_float2(c, s);
    }
}

__device__ __forceinline__ void rotate_with(float* lo, float* hi, const float2* tab, int i0) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        float2 cs = tab[i0 + k];
        float x0 = lo[k], x1 = hi[k];
        lo[k] = x0 * cs.x - x1 * cs.y;
        hi[k] = x1 * cs.x + x0 * cs.y;
    }
}

// =====================================================================================
// kvfix_rerope: streaming rotation of one plane.  grid = (tiles, chunks).
// =====================================================================================
constexpr int kRopeThreads = 256;
constexpr int kRopeItems = 4;  // pair vectors per thread

__global__ void __launch_bounds__(kRopeThreads)
rerope_kernel(const uint16_t* in, Plane p, uint16_t* out, Plane op,
              const int32_t* __restrict__ delta, RopeTheta th) {
    __shared__ float2 tab[kMaxHeadDim / 2];
    const int c = blockIdx.y;
    const int half = p.dim / 2;
    const int v16 = p.dim / 16;
    const int d = delta[c];
    build_table(tab, d, th, half, threadIdx.x, blockDim.x);
    __syncthreads();
    const long long items = (long long)p.layers * p.tokens * p.heads * v16;
    long long base = (long long)blockIdx.x * kRopeThreads * kRopeItems + threadIdx.x;
    uint4 lo[kRopeItems], hi[kRopeItems];
    long long off[kRopeItems], oof[kRopeItems];
#pragma unroll
    for (int k = 0; k < kRopeItems; ++k) {
        long long it = base + (long long)k * kRopeThreads;
        off[k] = -1;
        if (it < items) {
            int v = (int)(it % v16);
            long long r = it / v16;
            int h = (int)(r % p.heads);
            r /= p.heads;
            int t = (int)(r % p.tokens);
            int l = (int)(r / p.tokens);
            off[k] = p.row(c, l, t) + (long long)h * p.dim + 8 * v;
            oof[k] = op.row(c, l, t) + (long long)h * p.dim + 8 * v;
            lo[k] = ld_stream(reinterpret_cast<const uint4*>(in + off[k]));
            hi[k] = ld_stream(reinterpret_cast<const uint4*>(in + off[k] + half));
        }
    }
#pragma unroll
    for (int k = 0; k < kRopeItems; ++k) {
        if (off[k] < 0) continue;
        if (d != 0) {
            float a[8], b[8];
            unpack8(lo[k], a);
            unpack8(hi[k], b);
            int v = (int)((base + (long long)k * kRopeThreads) % v16);
            rotate_with(a, b, tab, 8 * v);
            lo[k] = pack8(a);
            hi[k] = pack8(b);
        }
        st_stream(reinterpret_cast<uint4*>(out + oof[k]), lo[k]);
        st_stream(reinterpret_cast<uint4*>(out + oof[k] + half), hi[k]);
    }
}

cudaError_t launch_rerope(const uint16_t* in, const kvfix_kv_desc& dd, uint16_t* out,
                          const kvfix_kv_desc& od, const int32_t* delta, const RopeTheta& th,
                          cudaStream_t s) {
    Plane p = plane_of(dd), op = plane_of(od);
    long long items = (long long)p.layers * p.tokens * p.heads * (p.dim / 16);
    if (items == 0 || p.chunks == 0) return cudaSuccess;
    long long tiles = (items + kRopeThreads * kRopeItems - 1) / (kRopeThreads * kRopeItems);
    for (int c0 = 0; c0 < p.chunks; c0 += 65535) {
        int nc = p.chunks - c0 < 65535 ? p.chunks - c0 : 65535;
        const uint16_t* qin = in + (long long)c0 * p.sc;
        uint16_t* qout = out + (long long)c0 * op.sc;
        dim3 grid((unsigned)tiles, (unsigned)nc);
        rerope_kernel<<<grid, kRopeThreads, 0, s>>>(qin, p, qout, op, delta + c0, th);
    }
    return cudaGetLastError();
}

// =====================================================================================
// Check-layer divergence for K and V of all agents: grid = (token tiles, R).
// One warp per token row; each lane owns pair vectors p = lane, lane+32, ...
// The reused row is loaded once and compared with every agent's fresh row.
// =====================================================================================
constexpr int kScoreWarps = 8;
constexpr int kScoreRowsPerWarp = 2;
constexpr int kAgentGroup = 8;

__global__ void __launch_bounds__(kScoreWarps * 32)
score_kernel(const uint16_t* __restrict__ k_reuse, const uint16_t* __restrict__ v_reuse, Plane rp,
             const uint16_t* __restrict__ k_fresh, const uint16_t* __restrict__ v_fresh, Plane fp,
             int agents, const int32_t* __restrict__ delta, RopeTheta th, float* __restrict__ d_k,
             float* __restrict__ d_v, float* __restrict__ w_k, float* __restrict__ w_v) {
    __shared__ float2 tab[kAgentGroup][kMaxHeadDim / 2];
    __shared__ int dl[kAgentGroup];
    const int R = rp.chunks;
    const int r = blockIdx.y;
    const int n = rp.tokens;
    const int half = rp.dim / 2;
    const int v16 = rp.dim / 16;
    const int P = rp.heads * v16;  // pair vectors per token row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t_base = blockIdx.x * (kScoreWarps * kScoreRowsPerWarp);
    const bool do_k = k_reuse != nullptr, do_v = v_reuse != nullptr;

    for (int a0 = 0; a0 < agents; a0 += kAgentGroup) {
        const int ag = agents - a0 < kAgentGroup ? agents - a0 : kAgentGroup;
        __syncthreads();
        for (int i = threadIdx.x; i < ag * half; i += blockDim.x) {
            int a = i / half, e = i % half;
            float c, s;
            rope_cos_sin(delta[(a0 + a) * R + r], th.theta[e], &c, &s);
            tab[a][e] = make_float2(c, s);
        }
        if (threadIdx.x < ag) dl[threadIdx.x] = delta[(a0 + threadIdx.x) * R + r];
        __syncthreads();
        for (int rr = 0; rr < kScoreRowsPerWarp; ++rr) {
            const int t = t_base + rr * kScoreWarps + warp;
            if (t >= n) continue;
            const long long ro = rp.row(r, 0, t);
            for (int a = 0; a < ag; ++a) {
                const int u = (a0 + a) * R + r;
                const long long fo = fp.row(u, 0, t);
                float sk = 0.f, sv = 0.f;
                for (int pv = lane; pv < P; pv += 32) {
                    const int h = pv / v16, v = pv % v16;
                    const long long eo = (long long)h * rp.dim + 8 * v;
                    if (do_k) {
                        float x0[8], x1[8], f0[8], f1[8];
                        unpack8(*reinterpret_cast<const uint4*>(k_reuse + ro + eo), x0);
                        unpack8(*reinterpret_cast<const uint4*>(k_reuse + ro + eo + half), x1);
                        unpack8(*reinterpret_cast<const uint4*>(k_fresh + fo + eo), f0);
                        unpack8(*reinterpret_cast<const uint4*>(k_fresh + fo + eo + half), f1);
                        if (dl[a] != 0) rotate_with(x0, x1, tab[a], 8 * v);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            float e0 = f0[q] - x0[q], e1 = f1[q] - x1[q];
                            sk = fmaf(e0, e0, sk);
                            sk = fmaf(e1, e1, sk);
                        }
                    }
                    if (do_v) {
                        float x0[8], x1[8], f0[8], f1[8];
                        unpack8(*reinterpret_cast<const uint4*>(v_reuse + ro + eo), x0);
                        unpack8(*reinterpret_cast<const uint4*>(v_reuse + ro + eo + half), x1);
                        unpack8(*reinterpret_cast<const uint4*>(v_fresh + fo + eo), f0);
                        unpack8(*reinterpret_cast<const uint4*>(v_fresh + fo + eo + half), f1);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            float e0 = f0[q] - x0[q], e1 = f1[q] - x1[q];
                            sv = fmaf(e0, e0, sv);
                            sv = fmaf(e1, e1, sv);
                        }
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    sk += __shfl_xor_sync(0xffffffffu, sk, o);
                    sv += __shfl_xor_sync(0xffffffffu, sv, o);
                }
                if (lane == 0) {
                    const long long oi = (long long)u * n + t;
                    if (do_k) {
                        float d = sqrtf(sk);
                        d_k[oi] = d;
                        w_k[oi] = fminf(d, 1.0f);
                    }
                    if (do_v) {
                        float d = sqrtf(sv);
                        d_v[oi] = d;
                        w_v[oi] = fminf(d, 1.0f);
                    }
                }
            }
        }
    }
}

cudaError_t launch_score(const uint16_t* k_reuse, const uint16_t* v_reuse,
                         const kvfix_kv_desc& reuse, const uint16_t* k_fresh,
                         const uint16_t* v_fresh, const kvfix_kv_desc& fresh, int agents,
                         const int32_t* delta, const RopeTheta& th, float* d_k, float* d_v,
                         float* w_k, float* w_v, cudaStream_t s) {
    Plane rp = plane_of(reuse), fp = plane_of(fresh);
    if (rp.tokens == 0 || rp.chunks == 0 || agents == 0) return cudaSuccess;
    const int rows = kScoreWarps * kScoreRowsPerWarp;
    dim3 grid((rp.tokens + rows - 1) / rows, rp.chunks);
    score_kernel<<<grid, kScoreWarps * 32, 0, s>>>(k_reuse, v_reuse, rp, k_fresh, v_fresh, fp,
                                                   agents, delta, th, d_k, d_v, w_k, w_v);
    return cudaGetLastError();
}

// =====================================================================================
// Block-wide top-b selection: the b largest keys, ties to the lower index.
// Radix select (8-bit digits, most significant first) finds the b-th largest key T;
// all keys > T are taken, and the lowest-index keys == T fill the rest.
// =====================================================================================
constexpr int kSelThreads = 1024;
constexpr int kSelSmemKeys = 16384;

// Order-preserving map of a float to an unsigned key (larger float -> larger key).
__device__ __forceinline__ uint32_t ordered_f32(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive scan of one int per thread over the block; returns the block total in *total.
__device__ int block_exclusive_scan(int x, int* warp_sums, int* total) {
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

template <typename Key>
struct SelectSmem {
    unsigned hist[256];
    int warp_sums[33];
    Key prefix;
    int remaining;
};

// Select into `bits` (n-bit bitmap in shared memory, cleared here) and write the
// ascending index list.  key_at(i) gives the key of index i.
template <typename Key, typename KeyAt>
__device__ void block_select(KeyAt key_at, int n, int b, uint32_t* bits, int32_t* idx_out,
                             SelectSmem<Key>& sm) {
    const int tid = threadIdx.x;
    const int words = (n + 31) / 32;
    for (int w = tid; w < words; w += blockDim.x) bits[w] = 0u;
    if (b <= 0) {
        __syncthreads();
        return;
    }
    constexpr int kBits = sizeof(Key) * 8;
    if (tid == 0) {
        sm.prefix = 0;
        sm.remaining = b;
    }
    __syncthreads();
    for (int shift = kBits - 8; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += blockDim.x) sm.hist[i] = 0u;
        __syncthreads();
        const Key prefix = sm.prefix;
        const Key hi_mask = (shift + 8 >= kBits) ? Key(0) : ~((Key(1) << (shift + 8)) - Key(1));
        for (int i = tid; i < n; i += blockDim.x) {
            Key k = key_at(i);
            if ((k & hi_mask) == (prefix & hi_mask)) atomicAdd(&sm.hist[(unsigned)(k >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 32) {
            // lane l holds bins 255-8l .. 248-8l (descending digit order)
            unsigned c[8];
            unsigned lsum = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                c[q] = sm.hist[255 - 8 * tid - q];
                lsum += c[q];
            }
            unsigned inc = lsum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                unsigned y = __shfl_up_sync(0xffffffffu, inc, o);
                if (tid >= o) inc += y;
            }
            unsigned before = inc - lsum;  // keys with a larger digit than this lane's bins
            const unsigned rem = (unsigned)sm.remaining;
            if (before < rem && rem <= inc) {
                unsigned acc = before;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (acc < rem && rem <= acc + c[q]) {
                        sm.prefix = prefix | (Key(255 - 8 * tid - q) << shift);
                        sm.remaining = (int)(rem - acc);
                    }
                    acc += c[q];
                }
            }
        }
        __syncthreads();
    }
    const Key T = sm.prefix;
    const int need_eq = sm.remaining;
    // Contiguous segment per thread, in index order.
    const int seg = (n + blockDim.x - 1) / blockDim.x;
    const int i0 = min(n, tid * seg), i1 = min(n, i0 + seg);
    int eq = 0;
    for (int i = i0; i < i1; ++i) eq += (key_at(i) == T);
    int tot;
    int eq_before = block_exclusive_scan(eq, sm.warp_sums, &tot);
    int cnt = 0;
    for (int i = i0; i < i1; ++i) {
        Key k = key_at(i);
        bool take = k > T;
        if (k == T) {
            take = eq_before < need_eq;
            ++eq_before;
        }
        if (take) {
            atomicOr(&bits[i >> 5], 1u << (i & 31));
            ++cnt;
        }
    }
    int out_before = block_exclusive_scan(cnt, sm.warp_sums, &tot);
    __syncthreads();
    for (int i = i0; i < i1; ++i) {
        if ((bits[i >> 5] >> (i & 31) & 1u) && out_before < b) idx_out[out_before++] = i;
    }
    __syncthreads();
}

// grid = units; dynamic smem: keys (when n fits) + 3 bitmaps.
__global__ void __launch_bounds__(kSelThreads)
select_f32_kernel(const float* __restrict__ d_k, const float* __restrict__ d_v, int n, int b,
                  int32_t* idx_k, int32_t* idx_v, uint32_t* mask_k, uint32_t* mask_v,
                  uint32_t* mask_union) {
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ SelectSmem<uint32_t> sm;
    const int words = (n + 31) / 32;
    uint32_t* bk = reinterpret_cast<uint32_t*>(dyn);
    uint32_t* bv = bk + words;
    uint32_t* keys = bv + words;
    const bool cached = n <= kSelSmemKeys;
    const long long u = blockIdx.x;
    for (int plane = 0; plane < 2; ++plane) {
        const float* d = plane == 0 ? d_k : d_v;
        uint32_t* bits = plane == 0 ? bk : bv;
        if (d == nullptr) {
            for (int w = threadIdx.x; w < words; w += blockDim.x) bits[w] = 0u;
            __syncthreads();
            continue;
        }
        const float* du = d + u * n;
        if (cached) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) keys[i] = ordered_f32(du[i]);
            __syncthreads();
            block_select<uint32_t>([&](int i) { return keys[i]; }, n, b, bits,
                                   (plane == 0 ? idx_k : idx_v) + u * b, sm);
        } else {
            block_select<uint32_t>([&](int i) { return ordered_f32(du[i]); }, n, b, bits,
                                   (plane == 0 ? idx_k : idx_v) + u * b, sm);
        }
        uint32_t* m = plane == 0 ? mask_k : mask_v;
        if (m)
            for (int w = threadIdx.x; w < words; w += blockDim.x) m[u * words + w] = bits[w];
        __syncthreads();
    }
    if (mask_union)
        for (int w = threadIdx.x; w < words; w += blockDim.x) mask_union[u * words + w] = bk[w] | bv[w];
}

cudaError_t launch_select_f32(const float* d_k, const float* d_v, int units, int n, int b,
                              int32_t* idx_k, int32_t* idx_v, uint32_t* mask_k,
                              uint32_t* mask_v, uint32_t* mask_union, cudaStream_t s) {
    if (units == 0 || n == 0) return cudaSuccess;
    const int words = (n + 31) / 32;
    size_t smem = sizeof(uint32_t) * (size_t)(2 * words + (n <= kSelSmemKeys ? n : 0));
    cudaError_t e = cudaFuncSetAttribute(select_f32_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    select_f32_kernel<<<units, kSelThreads, smem, s>>>(d_k, d_v, n, b, idx_k, idx_v, mask_k,
                                                       mask_v, mask_union);
    return cudaGetLastError();
}

// =====================================================================================
// Probe mean: one CTA per (unit, layer, head); 32 slots x (D/16) lanes.
// Slot g sums probes i = g, g+32, ... in order; slots are then added in order.
// The fresh probe rows are copied to the output on the way (they are the output).
// =====================================================================================
__global__ void probe_mean_kernel(const uint16_t* __restrict__ reuse, Plane rp,
                                  const uint16_t* __restrict__ fresh, Plane fp, uint16_t* out,
                                  Plane op, const int32_t* __restrict__ delta, RopeTheta th,
                                  int rotate, const int32_t* __restrict__ idx, int b,
                                  float* __restrict__ mu) {
    extern __shared__ __align__(16) float part[];  // [32][D]
    __shared__ float2 tab[kMaxHeadDim / 2];
    const int h = blockIdx.x, l = blockIdx.y, u = blockIdx.z;
    const int R = rp.chunks;
    const int r = u % R;
    const int D = rp.dim, half = D / 2, v16 = D / 16;
    const int n = rp.tokens;
    const int dlt = delta[u];
    const bool rot = rotate && dlt != 0;
    if (rot) build_table(tab, dlt, th, half, threadIdx.x, blockDim.x);
    __syncthreads();
    const int g = threadIdx.x / v16, v = threadIdx.x % v16;
    float acc0[8], acc1[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc0[k] = acc1[k] = 0.f;
    const int32_t* S = idx + (long long)u * b;
    const long long eo = (long long)h * D + 8 * v;
    for (int i = g; i < b; i += 32) {
        const int j = S[i];
        if (j < 0 || j >= n) {
            atomicOr(&g_status_repair, FLAG_BOUNDS);
            continue;
        }
        const long long ro = rp.row(r, l, j) + eo;
        const long long fo = fp.row(u, l, j) + eo;
        const long long oo = op.row(u, l, j) + eo;
        uint4 x0v = *reinterpret_cast<const uint4*>(reuse + ro);
        uint4 x1v = *reinterpret_cast<const uint4*>(reuse + ro + half);
        uint4 f0v = *reinterpret_cast<const uint4*>(fresh + fo);
        uint4 f1v = *reinterpret_cast<const uint4*>(fresh + fo + half);
        st_stream(reinterpret_cast<uint4*>(out + oo), f0v);
        st_stream(reinterpret_cast<uint4*>(out + oo + half), f1v);
        float x0[8], x1[8], f0[8], f1[8];
        unpack8(x0v, x0);
        unpack8(x1v, x1);
        unpack8(f0v, f0);
        unpack8(f1v, f1);
        if (rot) rotate_with(x0, x1, tab, 8 * v);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            acc0[k] += f0[k] - x0[k];
            acc1[k] += f1[k] - x1[k];
        }
    }
    float* mine = part + g * D;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        mine[8 * v + k] = acc0[k];
        mine[half + 8 * v + k] = acc1[k];
    }
    __syncthreads();
    float* mu_row = mu + ((long long)u * rp.layers + l) * ((long long)rp.heads * D) + (long long)h * D;
    for (int e = threadIdx.x; e < D; e += blockDim.x) {
        float s = 0.f;
        for (int q = 0; q < 32; ++q) s += part[q * D + e];
        mu_row[e] = b > 0 ? s / (float)b : 0.f;
    }
}

// =====================================================================================
// Correction of the non-probe rows: one CTA per (token tile, layer, reused chunk).
// The reused tile is read once; every agent's corrected rows are written from it.
// =====================================================================================
constexpr int kCorrThreads = 256;
constexpr int kCorrTile = 64;  // tokens per CTA

__global__ void __launch_bounds__(kCorrThreads)
correct_kernel(const uint16_t* __restrict__ reuse, Plane rp, uint16_t* out, Plane op, int agents,
               const int32_t* __restrict__ delta, RopeTheta th, int rotate,
               const int32_t* __restrict__ idx, int b, const float* __restrict__ w,
               const float* __restrict__ mu) {
    extern __shared__ __align__(16) float smu[];  // [kAgentGroup][H*D]
    __shared__ float2 tab[kAgentGroup][kMaxHeadDim / 2];
    __shared__ uint32_t member[kAgentGroup][kCorrTile / 32];
    __shared__ float sw[kAgentGroup][kCorrTile];
    __shared__ int rot_on[kAgentGroup];
    const int t0 = blockIdx.x * kCorrTile, l = blockIdx.y, r = blockIdx.z;
    const int R = rp.chunks, n = rp.tokens;
    const int D = rp.dim, half = D / 2, v16 = D / 16, HD = rp.heads * D;
    const int P = rp.heads * v16;
    const int tt = min(kCorrTile, n - t0);
    const int items = tt * P;

    for (int a0 = 0; a0 < agents; a0 += kAgentGroup) {
        const int ag = min(kAgentGroup, agents - a0);
        __syncthreads();
        for (int i = threadIdx.x; i < ag * (kCorrTile / 32); i += blockDim.x)
            member[i / (kCorrTile / 32)][i % (kCorrTile / 32)] = 0u;
        for (int i = threadIdx.x; i < ag * half; i += blockDim.x) {
            int a = i / half, e = i % half;
            float c = 1.f, s = 0.f;
            if (rotate) rope_cos_sin(delta[(a0 + a) * R + r], th.theta[e], &c, &s);
            tab[a][e] = make_float2(c, s);
        }
        if (threadIdx.x < ag) rot_on[threadIdx.x] = rotate && delta[(a0 + threadIdx.x) * R + r] != 0;
        for (int i = threadIdx.x; i < ag * HD; i += blockDim.x) {
            int a = i / HD, e = i % HD;
            const long long u = (long long)(a0 + a) * R + r;
            smu[i] = b > 0 ? mu[(u * rp.layers + l) * HD + e] : 0.f;
        }
        for (int i = threadIdx.x; i < ag * tt; i += blockDim.x) {
            int a = i / tt, t = i % tt;
            const long long u = (long long)(a0 + a) * R + r;
            sw[a][t] = w[u * n + t0 + t];
        }
        __syncthreads();
        for (int i = threadIdx.x; i < ag * b; i += blockDim.x) {
            int a = i / b, q = i % b;
            const long long u = (long long)(a0 + a) * R + r;
            int j = idx[u * b + q];
            if (j >= t0 && j < t0 + tt) atomicOr(&member[a][(j - t0) >> 5], 1u << ((j - t0) & 31));
        }
        __syncthreads();
        for (int it = threadIdx.x; it < items; it += kCorrThreads) {
            const int t = it / P, pv = it % P;
            const int h = pv / v16, v = pv % v16;
            const long long eo = (long long)h * D + 8 * v;
            const long long ro = rp.row(r, l, t0 + t) + eo;
            const uint4 x0v = ld_stream(reinterpret_cast<const uint4*>(reuse + ro));
            const uint4 x1v = ld_stream(reinterpret_cast<const uint4*>(reuse + ro + half));
            for (int a = 0; a < ag; ++a) {
                if (member[a][t >> 5] >> (t & 31) & 1u) continue;
                float x0[8], x1[8];
                unpack8(x0v, x0);
                unpack8(x1v, x1);
                if (rot_on[a]) rotate_with(x0, x1, tab[a], 8 * v);
                if (b > 0) {
                    const float wt = sw[a][t];
                    const float* m = smu + a * HD + h * D + 8 * v;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        x0[k] = fmaf(wt, m[k], x0[k]);
                        x1[k] = fmaf(wt, m[half + k], x1[k]);
                    }
                }
                const long long u = (long long)(a0 + a) * R + r;
                const long long oo = op.row((int)u, l, t0 + t) + eo;
                st_stream(reinterpret_cast<uint4*>(out + oo), pack8(x0));
                st_stream(reinterpret_cast<uint4*>(out + oo + half), pack8(x1));
            }
        }
    }
}

cudaError_t launch_mean_correct(const uint16_t* reuse, const kvfix_kv_desc& rd,
                                const uint16_t* fresh, const kvfix_kv_desc& fd, uint16_t* out,
                                const kvfix_kv_desc& od, int agents, const int32_t* delta,
                                const RopeTheta& th, bool rotate, const int32_t* idx, int b,
                                const float* w, float* mu, cudaStream_t s) {
    Plane rp = plane_of(rd), fp = plane_of(fd), op = plane_of(od);
    const int units = agents * rp.chunks;
    if (units == 0 || rp.layers == 0 || rp.tokens == 0) return cudaSuccess;
    const size_t mu_bytes = sizeof(float) * (size_t)units * rp.layers * rp.heads * rp.dim;
    cudaError_t e;
    if (b > 0) {
        dim3 grid(rp.heads, rp.layers, units);
        size_t smem = sizeof(float) * 32 * (size_t)rp.dim;
        probe_mean_kernel<<<grid, 2 * rp.dim, smem, s>>>(reuse, rp, fresh, fp, out, op, delta, th,
                                                         rotate ? 1 : 0, idx, b, mu);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    } else {
        if ((e = cudaMemsetAsync(mu, 0, mu_bytes, s)) != cudaSuccess) return e;
    }
    dim3 grid((rp.tokens + kCorrTile - 1) / kCorrTile, rp.layers, rp.chunks);
    size_t smem = sizeof(float) * kAgentGroup * (size_t)rp.heads * rp.dim;
    e = cudaFuncSetAttribute(correct_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    correct_kernel<<<grid, kCorrThreads, smem, s>>>(reuse, rp, out, op, agents, delta, th,
                                                    rotate ? 1 : 0, idx, b, w, mu);
    return cudaGetLastError();
}

}  // namespace kvfix
