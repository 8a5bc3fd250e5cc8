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
#include <string.h>


#include "common.cuh"
#include "tc.cuh"

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
        lo[k] = __fmaf_rn(x0, cs.x, __fmul_rn(x1, -cs.y));  // same rounding as the packed form
        hi[k] = __fmaf_rn(x1, cs.x, __fmul_rn(x0, cs.y));
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
// One warp per (token row, plane): warps 2w and 2w+1 of a CTA take the K and V rows of
// the same token.  Each lane owns pair vectors p = lane, lane+32, ... and loads two of
// them at a time, so a row of up to 64 pair vectors costs one memory round trip.
// =====================================================================================
constexpr int kScoreWarps = 8;
constexpr int kScoreRowsPerCta = kScoreWarps / 2;
constexpr int kAgentGroup = 8;

__device__ __forceinline__ float sq_diff8(const uint4& x, const uint4& f, float acc) {
    float xf[8], ff[8];
    unpack8(x, xf);
    unpack8(f, ff);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float e = ff[q] - xf[q];
        acc = fmaf(e, e, acc);
    }
    return acc;
}

// Reused and fresh pieces of two pair vectors of one token row (the second may be absent).
struct ScorePv2 {
    uint4 x0a, x1a, f0a, f1a, x0b, x1b, f0b, f1b;
};

__device__ __forceinline__ ScorePv2 score_load(const uint16_t* reuse, long long ro, const uint16_t* fresh,
                                               long long fo, long long e0, long long e1, int half) {
    ScorePv2 v;
    v.x0a = *reinterpret_cast<const uint4*>(reuse + ro + e0);
    v.x1a = *reinterpret_cast<const uint4*>(reuse + ro + e0 + half);
    v.f0a = *reinterpret_cast<const uint4*>(fresh + fo + e0);
    v.f1a = *reinterpret_cast<const uint4*>(fresh + fo + e0 + half);
    v.x0b = *reinterpret_cast<const uint4*>(reuse + ro + e1);
    v.x1b = *reinterpret_cast<const uint4*>(reuse + ro + e1 + half);
    v.f0b = *reinterpret_cast<const uint4*>(fresh + fo + e1);
    v.f1b = *reinterpret_cast<const uint4*>(fresh + fo + e1 + half);
    return v;
}

__device__ __forceinline__ float score_rot8(const uint4& x0v, const uint4& x1v, const uint4& f0v, const uint4& f1v,
                                            const float2* tab, int i0, float ss) {
    float x0[8], x1[8], f0[8], f1[8];
    unpack8(x0v, x0);
    unpack8(x1v, x1);
    unpack8(f0v, f0);
    unpack8(f1v, f1);
    rotate_with(x0, x1, tab, i0);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float e0 = f0[q] - x0[q], e1 = f1[q] - x1[q];
        ss = fmaf(e0, e0, ss);
        ss = fmaf(e1, e1, ss);
    }
    return ss;
}

__global__ void __launch_bounds__(kScoreWarps * 32)
score_kernel(const uint16_t* __restrict__ k_reuse, const uint16_t* __restrict__ v_reuse, Plane rp,
             const uint16_t* __restrict__ k_fresh, const uint16_t* __restrict__ v_fresh, Plane fp,
             int agents, const int32_t* __restrict__ delta, RopeTheta th, float* __restrict__ d_k,
             float* __restrict__ d_v, float* __restrict__ w_k, float* __restrict__ w_v,
             uint32_t* mask_union) {
    __shared__ float2 tab[kAgentGroup][kMaxHeadDim / 2];
    __shared__ int dl[kAgentGroup];
    const int R = rp.chunks;
    const int r = blockIdx.y;
    const int n = rp.tokens;
    const int half = rp.dim / 2;
    const int v16 = rp.dim / 16;
    const int P = rp.heads * v16;  // pair vectors per token row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool keys = (warp & 1) == 0;
    const uint16_t* reuse = keys ? k_reuse : v_reuse;
    const uint16_t* fresh = keys ? k_fresh : v_fresh;
    float* d_out = keys ? d_k : d_v;
    float* w_out = keys ? w_k : w_v;
    const int t_base = blockIdx.x * kScoreRowsPerCta;
    const int t = t_base + (warp >> 1);
    const bool row_ok = reuse != nullptr && t < n;
    const long long ro = row_ok ? rp.row(r, 0, t) : 0;
    auto offs = [&](int p0, long long& e0, long long& e1) {  // element offsets of p0 and p0 + 32
        const int p1 = p0 + 32 < P ? p0 + 32 : p0;
        e0 = (long long)(p0 / v16) * rp.dim + 8 * (p0 % v16);
        e1 = (long long)(p1 / v16) * rp.dim + 8 * (p1 % v16);
    };
    pdl_trigger();  // the selection may launch; it waits for these scores
    if (mask_union) {  // the selection ORs both planes into it afterwards
        const int words = (n + 31) / 32;
        const int w0 = t_base / 32, w1 = min(words, (t_base + kScoreRowsPerCta + 31) / 32);
        for (int i = threadIdx.x; i < agents * (w1 - w0); i += blockDim.x) {
            const int a = i / (w1 - w0), w = w0 + i % (w1 - w0);
            mask_union[((long long)a * R + r) * words + w] = 0u;
        }
    }

    for (int a0 = 0; a0 < agents; a0 += kAgentGroup) {
        const int ag = agents - a0 < kAgentGroup ? agents - a0 : kAgentGroup;
        __syncthreads();
        // The first agent's first two pair vectors are requested before the angle table is
        // built, so the table's arithmetic overlaps the memory round trip.
        ScorePv2 v;
        if (row_ok && lane < P) {
            long long e0, e1;
            offs(lane, e0, e1);
            v = score_load(reuse, ro, fresh, fp.row(a0 * R + r, 0, t), e0, e1, half);
        }
        if (k_reuse != nullptr)
            for (int i = threadIdx.x; i < ag * half; i += blockDim.x) {
                int a = i / half, e = i % half;
                float c, s;
                rope_cos_sin(delta[(a0 + a) * R + r], th.theta[e], &c, &s);
                tab[a][e] = make_float2(c, s);
            }
        if (threadIdx.x < ag) dl[threadIdx.x] = delta[(a0 + threadIdx.x) * R + r];
        __syncthreads();
        if (!row_ok) continue;
        for (int a = 0; a < ag; ++a) {
            const int u = (a0 + a) * R + r;
            const long long fo = fp.row(u, 0, t);
            const bool rot = keys && dl[a] != 0;
            float ss = 0.f;
            for (int p0 = lane; p0 < P; p0 += 64) {
                const bool two = p0 + 32 < P;
                long long e0, e1;
                offs(p0, e0, e1);
                if (a > 0 || p0 != lane) v = score_load(reuse, ro, fresh, fo, e0, e1, half);
                if (rot) {
                    ss = score_rot8(v.x0a, v.x1a, v.f0a, v.f1a, tab[a], 8 * (p0 % v16), ss);
                    if (two) ss = score_rot8(v.x0b, v.x1b, v.f0b, v.f1b, tab[a], 8 * ((p0 + 32) % v16), ss);
                } else {
                    ss = sq_diff8(v.x0a, v.f0a, ss);
                    ss = sq_diff8(v.x1a, v.f1a, ss);
                    if (two) {
                        ss = sq_diff8(v.x0b, v.f0b, ss);
                        ss = sq_diff8(v.x1b, v.f1b, ss);
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (lane == 0) {
                const long long oi = (long long)u * n + t;
                const float d = sqrtf(ss);
                d_out[oi] = d;
                w_out[oi] = fminf(d, 1.0f);
            }
        }
    }
}

cudaError_t launch_score(const uint16_t* k_reuse, const uint16_t* v_reuse,
                         const kvfix_kv_desc& reuse, const uint16_t* k_fresh,
                         const uint16_t* v_fresh, const kvfix_kv_desc& fresh, int agents,
                         const int32_t* delta, const RopeTheta& th, float* d_k, float* d_v,
                         float* w_k, float* w_v, uint32_t* mask_union, cudaStream_t s) {
    Plane rp = plane_of(reuse), fp = plane_of(fresh);
    if (rp.tokens == 0 || rp.chunks == 0 || agents == 0) return cudaSuccess;
    dim3 grid((rp.tokens + kScoreRowsPerCta - 1) / kScoreRowsPerCta, rp.chunks);
    score_kernel<<<grid, kScoreWarps * 32, 0, s>>>(k_reuse, v_reuse, rp, k_fresh, v_fresh, fp,
                                                   agents, delta, th, d_k, d_v, w_k, w_v, mask_union);
    return cudaGetLastError();
}

// =====================================================================================
// Block-wide top-b selection: the b largest keys, ties to the lower index.
// Radix select, most significant bits first.  The bits above the highest bit in which
// the block's smallest and largest keys differ are shared by every key and settled at
// once; the rest are settled 8 at a time, each pass a histogram of the keys that still
// match the settled prefix.  The result T is the b-th largest key: every key > T is
// taken, and the lowest-index keys == T fill the rest.
// =====================================================================================
constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelSmemKeys = 16384;

// Order-preserving map of a float to an unsigned key (larger float -> larger key).
__device__ __forceinline__ uint32_t ordered_f32(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SelectSmem {
    unsigned hist[2][256];  // one histogram per pass parity
    uint32_t wmin[kSelWarps], wmax[kSelWarps];
    int wgt[kSelWarps], weq[kSelWarps];
    uint32_t prefix[2];
    int remaining[2];
};

// Select into `bits` (n-bit bitmap in shared memory, cleared here) and write the
// ascending index list.  key_at(i) gives the key of index i.  blockDim.x == kSelThreads.
template <typename KeyAt>
__device__ void block_select(KeyAt key_at, int n, int b, uint32_t* bits, int32_t* idx_out, SelectSmem& sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned full = 0xffffffffu;
    const int words = (n + 31) / 32;
    for (int w = tid; w < words; w += kSelThreads) bits[w] = 0u;
    if (tid < 256) sm.hist[0][tid] = 0u;
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int i = tid; i < n; i += kSelThreads) {
        const uint32_t k = key_at(i);
        kmin = min(kmin, k);
        kmax = max(kmax, k);
    }
    kmin = __reduce_min_sync(full, kmin);
    kmax = __reduce_max_sync(full, kmax);
    if (lane == 0) {
        sm.wmin[warp] = kmin;
        sm.wmax[warp] = kmax;
    }
    __syncthreads();
    if (b <= 0) return;
    kmin = __reduce_min_sync(full, sm.wmin[lane]);
    kmax = __reduce_max_sync(full, sm.wmax[lane]);
    int hi = kmin == kmax ? 0 : 32 - __clz(kmin ^ kmax);  // bits [0, hi) are still open
    uint32_t prefix = hi == 32 ? 0u : (kmax >> hi) << hi;
    int remaining = b;  // keys still to take among those matching the prefix
    for (int pass = 0; hi > 0; ++pass) {
        const int wdt = hi < 8 ? hi : 8, shift = hi - wdt;
        unsigned* h = sm.hist[pass & 1];
        // histogram of the digits of the keys that match the prefix (plain shared atomics)
        for (int i0 = 0; i0 < n; i0 += kSelThreads) {
            const int i = i0 + tid;
            unsigned dig = 256u;  // not counted
            if (i < n) {
                const uint32_t k = key_at(i);
                if (hi == 32 || (k >> hi) == (prefix >> hi)) dig = (k >> shift) & ((1u << wdt) - 1u);
            }
            if (dig < 256u) atomicAdd(&h[dig], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l holds bins 255-8l .. 248-8l (descending digit order)
            unsigned c[8], lsum = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                c[q] = h[255 - 8 * lane - q];
                lsum += c[q];
            }
            unsigned inc = lsum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_up_sync(full, inc, o);
                if (lane >= o) inc += y;
            }
            const unsigned before = inc - lsum;  // keys with a larger digit than this lane's bins
            const unsigned rem = (unsigned)remaining;
            if (before < rem && rem <= inc) {
                unsigned acc = before;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (acc < rem && rem <= acc + c[q]) {
                        sm.prefix[pass & 1] = prefix | ((uint32_t)(255 - 8 * lane - q) << shift);
                        sm.remaining[pass & 1] = (int)(rem - acc);
                    }
                    acc += c[q];
                }
            }
        } else if (tid - 32 < 256) {
            sm.hist[(pass + 1) & 1][tid - 32] = 0u;  // the next pass's histogram
        }
        __syncthreads();
        prefix = sm.prefix[pass & 1];
        remaining = sm.remaining[pass & 1];
        hi = shift;
    }
    const uint32_t T = prefix;
    // Keys > T and == T on this thread's contiguous segment, then one block scan of both.
    const int seg = (n + kSelThreads - 1) / kSelThreads;
    const int i0 = min(n, tid * seg), i1 = min(n, i0 + seg);
    int gt = 0, eq = 0;
    for (int i = i0; i < i1; ++i) {
        const uint32_t k = key_at(i);
        gt += k > T;
        eq += k == T;
    }
    int igt = gt, ieq = eq;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yg = __shfl_up_sync(full, igt, o), ye = __shfl_up_sync(full, ieq, o);
        if (lane >= o) {
            igt += yg;
            ieq += ye;
        }
    }
    if (lane == 31) {
        sm.wgt[warp] = igt;
        sm.weq[warp] = ieq;
    }
    __syncthreads();
    int wg = sm.wgt[lane], we = sm.weq[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yg = __shfl_up_sync(full, wg, o), ye = __shfl_up_sync(full, we, o);
        if (lane >= o) {
            wg += yg;
            we += ye;
        }
    }
    // exclusive offsets of this warp
    const int og = warp ? __shfl_sync(full, wg, warp - 1) : 0;
    const int oe = warp ? __shfl_sync(full, we, warp - 1) : 0;
    const int gt_before = og + igt - gt;
    int eq_seen = oe + ieq - eq;
    int out = gt_before + min(eq_seen, remaining);
    for (int i = i0; i < i1; ++i) {
        const uint32_t k = key_at(i);
        bool take = k > T;
        if (k == T) {
            take = eq_seen < remaining;
            ++eq_seen;
        }
        if (take) {
            idx_out[out++] = i;
            atomicOr(&bits[i >> 5], 1u << (i & 31));
        }
    }
    __syncthreads();
}

// grid = (units, 2 planes); dynamic smem: keys (when n fits) + one bitmap.  The union
// mask (zeroed by the score kernel) receives both planes' bits with atomicOr.
__global__ void __launch_bounds__(kSelThreads)
select_f32_kernel(const float* __restrict__ d_k, const float* __restrict__ d_v, int n, int b,
                  int32_t* idx_k, int32_t* idx_v, uint32_t* mask_k, uint32_t* mask_v,
                  uint32_t* mask_union) {
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ SelectSmem sm;
    const int words = (n + 31) / 32;
    uint32_t* bits = reinterpret_cast<uint32_t*>(dyn);
    uint32_t* keys = bits + words;
    const bool cached = n <= kSelSmemKeys;
    const long long u = blockIdx.x;
    const int plane = blockIdx.y;
    pdl_wait();     // scores of the score kernel
    pdl_trigger();  // the correction may launch; it waits for these probe sets
    const float* d = plane == 0 ? d_k : d_v;
    if (d == nullptr) return;
    const float* du = d + u * n;
    int32_t* idx_out = (plane == 0 ? idx_k : idx_v) + u * b;
    if (cached) {
        for (int i = threadIdx.x; i < n; i += blockDim.x) keys[i] = ordered_f32(du[i]);
        __syncthreads();
        block_select([&](int i) { return keys[i]; }, n, b, bits, idx_out, sm);
    } else {
        block_select([&](int i) { return ordered_f32(du[i]); }, n, b, bits, idx_out, sm);
    }
    uint32_t* m = plane == 0 ? mask_k : mask_v;
    if (m)
        for (int w = threadIdx.x; w < words; w += blockDim.x) m[u * words + w] = bits[w];
    if (mask_union)
        for (int w = threadIdx.x; w < words; w += blockDim.x)
            if (bits[w]) atomicOr(&mask_union[u * words + w], bits[w]);
}

cudaError_t launch_select_f32(const float* d_k, const float* d_v, int units, int n, int b,
                              int32_t* idx_k, int32_t* idx_v, uint32_t* mask_k,
                              uint32_t* mask_v, uint32_t* mask_union, cudaStream_t s) {
    if (units == 0 || n == 0) return cudaSuccess;
    const int words = (n + 31) / 32;
    size_t smem = sizeof(uint32_t) * (size_t)(words + (n <= kSelSmemKeys ? n : 0));
    cudaError_t e = cudaFuncSetAttribute(select_f32_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_chained(select_f32_kernel, dim3(units, 2), dim3(kSelThreads), smem, s, d_k, d_v, n, b,
                          idx_k, idx_v, mask_k, mask_v, mask_union);
}

// =====================================================================================
// Probe-mean correction: two kernels chained by programmatic dependent launch.  Both
// work on column slices of the token row: `cw` consecutive row elements made of whole
// heads (128 elements unless a head is wider), so an 8 x 128 row has eight slices.
//   probe_mean_kernel: one CTA per (unit, layer, plane, slice).  Thread (s, quad pair)
//     sums the probes i = s, s + 32, ... of slot s in probe-list order, the loads of
//     four rows in flight at a time; fresh and reused rows are summed separately and
//     the reused sum is rotated once, P_s = sum(fresh) - rot(sum(reuse)) (the rotation
//     is linear).  The fresh probe rows are copied to the output on the way.  The CTA
//     then adds the group sums Q_g = ((P_4g + P_4g+1) + P_4g+2) + P_4g+3 in order
//     g = 0..7 and divides by b: the mean, written to the mean output.
//   mean_stream_kernel: one CTA per (row block, layer, plane, slice, reused chunk,
//     agent group) streams the block's reused rows through a 3-stage ring of 16 KB
//     shared-memory tiles, each one TMA tensor copy of (cw columns x TR rows) completed
//     in bytes on a "full" mbarrier and released by every warp on an "empty" mbarrier.
//     Each reused row is read once and the corrected row of every agent of the group is
//     written from it; probe rows are skipped (the mean kernel wrote them).  The
//     barriers, the rotation table and the first tiles are set up before the wait on
//     the mean kernel.
// Work unit of a thread: a "quad pair" -- dims [4v, 4v+4) of one head and their rotation
// partners [D/2+4v, D/2+4v+4) -- so the rotation never leaves the thread.  The summation
// order is fixed per element and shared with the multi-agent kernels below: one call
// for N agents is bit-identical to N calls, whatever the slicing.
// =====================================================================================
constexpr int kGroups = 8;         // the 32 probe slots fold in 8 groups of 4
constexpr int kSlotsPerGroup = 4;
constexpr int kSlots = kGroups * kSlotsPerGroup;
constexpr int kMcSliceCols = 128;  // width of a column slice in elements (whole heads)
constexpr int kPmBatch = 2;        // probe rows of a slot whose loads are in flight together
constexpr int kMsThreads = 256;
constexpr int kMsWarps = kMsThreads / 32;
constexpr int kMsStages = 3;
constexpr int kMsTileBytes = 16384;
constexpr int kMsRows = 512;       // rows per CTA of the stream kernel

struct McMaps {  // TMA maps of the two reused planes (dims: row elements, tokens, layers, chunks)
    CUtensorMap reuse[2];
};

struct McArgs {
    const uint16_t* reuse[2];
    const uint16_t* fresh[2];
    uint16_t* out[2];
    const int32_t* idx[2];
    const float* w[2];
    float* mu[2];
    Plane rp, fp, op;
    int agents, b, rows_per_cta, tile_rows, cw, slices;
    const int32_t* delta;
    RopeTheta th;
};

__global__ void __launch_bounds__(1024, 1) probe_mean_kernel(McArgs args) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float2 tab[kMaxHeadDim / 2];
    const int slice = blockIdx.x, plane = blockIdx.y & 1, l = blockIdx.y >> 1, u = blockIdx.z;
    const uint16_t* reuse = args.reuse[plane];
    if (reuse == nullptr) return;
    const uint16_t* fresh = args.fresh[plane];
    uint16_t* out = args.out[plane];
    const Plane& rp = args.rp;
    const Plane& fp = args.fp;
    const Plane& op = args.op;
    const int R = rp.chunks, r = u % R, n = rp.tokens, L = rp.layers;
    const int D = rp.dim, half = D / 2, v8 = D / 8;
    const int HD = rp.heads * D, CW = args.cw, c0 = slice * CW, P = CW / 8;
    const int b = args.b;
    const int tid = threadIdx.x, nthreads = blockDim.x;  // kSlots * P threads
    float* Ps = reinterpret_cast<float*>(smem);  // [32 slots][CW], natural element order
    const int dl = args.delta[u];
    const bool rot = plane == 0 && dl != 0;
    if (rot)  // independent of the selection: before the wait
        for (int e = tid; e < half; e += nthreads) {
            float c, s;
            rope_cos_sin(dl, args.th.theta[e], &c, &s);
            tab[e] = make_float2(c, s);
        }
    // The stream kernel may launch now: it sets up its ring and first tiles while this
    // grid runs, and waits for this grid's completion before it reads the means.
    pdl_trigger();
    pdl_wait();  // probe sets of the selection kernel
    float* mu_g = args.mu[plane] + ((long long)u * L + l) * HD + c0;
    if (b == 0) {
        for (int e = tid; e < CW; e += nthreads) mu_g[e] = 0.f;
        return;
    }
    const int s = tid / P, pq = tid % P;
    const int h = pq / v8, v = pq % v8;
    const int eo = c0 + h * D + 4 * v;
    const int32_t* S = args.idx[plane] + (long long)u * b;
    float fs0[4], fs1[4], xs0[4], xs1[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) fs0[k] = fs1[k] = xs0[k] = xs1[k] = 0.f;
    auto probe = [&](int i) {  // row index of list position i, or -1 (past the end or out of range)
        if (i >= b) return -1;
        const int j = __ldg(S + i);
        if (j < 0 || j >= n) {
            atomicOr(&g_status_repair, FLAG_BOUNDS);
            return -1;
        }
        return j;
    };
    int jn[kPmBatch];
#pragma unroll
    for (int q = 0; q < kPmBatch; ++q) jn[q] = probe(s + kSlots * q);
    for (int i0 = s; i0 < b; i0 += kSlots * kPmBatch) {
        int jj[kPmBatch];
        uint2 xv[kPmBatch][2], fv[kPmBatch][2];
#pragma unroll
        for (int q = 0; q < kPmBatch; ++q) {
            jj[q] = jn[q];
            if (jj[q] >= 0) {
                const long long ro = rp.row(r, l, jj[q]) + eo;
                const long long fo = fp.row(u, l, jj[q]) + eo;
                xv[q][0] = __ldg(reinterpret_cast<const uint2*>(reuse + ro));
                xv[q][1] = __ldg(reinterpret_cast<const uint2*>(reuse + ro + half));
                fv[q][0] = __ldcs(reinterpret_cast<const uint2*>(fresh + fo));
                fv[q][1] = __ldcs(reinterpret_cast<const uint2*>(fresh + fo + half));
            }
        }
#pragma unroll
        for (int q = 0; q < kPmBatch; ++q) jn[q] = probe(i0 + kSlots * (kPmBatch + q));  // the next batch
#pragma unroll
        for (int q = 0; q < kPmBatch; ++q) {  // in list order
            if (jj[q] < 0) continue;
            const long long oo = op.row(u, l, jj[q]) + eo;
            __stcs(reinterpret_cast<uint2*>(out + oo), fv[q][0]);
            __stcs(reinterpret_cast<uint2*>(out + oo + half), fv[q][1]);
            add4(xv[q][0], xs0);
            add4(xv[q][1], xs1);
            add4(fv[q][0], fs0);
            add4(fv[q][1], fs1);
        }
    }
    __syncthreads();  // the angle table
    if (rot) {
        float c[4], sn[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 cs = tab[4 * v + k];
            c[k] = cs.x;
            sn[k] = cs.y;
        }
        rotate4(xs0, xs1, c, sn);
    }
    float* mine = Ps + s * CW + (eo - c0);
    *reinterpret_cast<float4*>(mine) =
        make_float4(fs0[0] - xs0[0], fs0[1] - xs0[1], fs0[2] - xs0[2], fs0[3] - xs0[3]);
    *reinterpret_cast<float4*>(mine + half) =
        make_float4(fs1[0] - xs1[0], fs1[1] - xs1[1], fs1[2] - xs1[2], fs1[3] - xs1[3]);
    __syncthreads();
    for (int e = tid; e < CW; e += nthreads) {
        float sum = 0.f;
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
            const float* q = Ps + (kSlotsPerGroup * g) * CW + e;
            sum += ((q[0] + q[CW]) + q[2 * CW]) + q[3 * CW];
        }
        mu_g[e] = sum / (float)b;
    }
}

// One quad pair of one non-probe row: rotate (keys, delta != 0), add w * mean, round to
// bf16 and store.  The same packed f32x2 arithmetic as the multi-agent stream kernel.
struct McConst {  // per-agent constants of a quad pair: cos, sin, -sin, mean (lo, hi)
    float2 c2[2], s2[2], ns2[2], m0[2], m1[2];
};

__device__ __forceinline__ void correct_quad_pair(const uint16_t* tr, uint16_t* o, int half, bool rot, bool add,
                                                  float wt, const McConst& k) {
    const uint2 lo_raw = *reinterpret_cast<const uint2*>(tr);
    const uint2 hi_raw = *reinterpret_cast<const uint2*>(tr + half);
    float2 x0[2], x1[2];
    x0[0] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&lo_raw.x));
    x0[1] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&lo_raw.y));
    x1[0] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hi_raw.x));
    x1[1] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hi_raw.y));
    if (rot) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float2 lo = __ffma2_rn(x0[q], k.c2[q], __fmul2_rn(x1[q], k.ns2[q]));
            const float2 hi = __ffma2_rn(x1[q], k.c2[q], __fmul2_rn(x0[q], k.s2[q]));
            x0[q] = lo;
            x1[q] = hi;
        }
    }
    if (add) {
        const float2 w2 = make_float2(wt, wt);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            x0[q] = __ffma2_rn(w2, k.m0[q], x0[q]);
            x1[q] = __ffma2_rn(w2, k.m1[q], x1[q]);
        }
    }
    uint2 lo_out, hi_out;
    *reinterpret_cast<__nv_bfloat162*>(&lo_out.x) = __float22bfloat162_rn(x0[0]);
    *reinterpret_cast<__nv_bfloat162*>(&lo_out.y) = __float22bfloat162_rn(x0[1]);
    *reinterpret_cast<__nv_bfloat162*>(&hi_out.x) = __float22bfloat162_rn(x1[0]);
    *reinterpret_cast<__nv_bfloat162*>(&hi_out.y) = __float22bfloat162_rn(x1[1]);
    st_stream2(reinterpret_cast<uint2*>(o), lo_out);
    st_stream2(reinterpret_cast<uint2*>(o + half), hi_out);
}

struct MsLayout {  // byte offsets into the stream kernel's dynamic shared memory
    int ring, mu, cs, member, wts, total, words;
};

__host__ __device__ inline MsLayout ms_layout(int CW, int half, int ag, int rows, int tile_rows) {
    MsLayout m;
    m.ring = 0;
    m.mu = kMsStages * tile_rows * CW * 2;  // [ag][CW] means, natural order
    m.cs = m.mu + 4 * ag * CW;               // [ag][half] (cos, sin)
    m.member = m.cs + 8 * ag * half;          // [ag][words] probe bits of the block's rows
    m.words = (rows + 31) / 32;
    m.wts = m.member + 4 * ag * m.words;      // [ag][rows] weights
    m.total = m.wts + 4 * ag * rows;
    return m;
}

// kCW: the slice width when it is known at compile time (the row loop then unrolls), else 0.
template <int kCW>
__global__ void __launch_bounds__(kMsThreads, 4)
mean_stream_kernel(const __grid_constant__ McMaps maps, McArgs args) {
    // TMA tile copies need a 128-byte aligned destination: the ring gets a symbol of its own
    extern __shared__ __align__(1024) unsigned char ms_smem[];
    unsigned char* smem = ms_smem;
    __shared__ __align__(8) uint64_t full[kMsStages];
    __shared__ __align__(8) uint64_t empty[kMsStages];
    __shared__ int rot_on[kAgentGroup];
    __shared__ int abort_flag;
    const int slice = (int)blockIdx.y % args.slices, lp = (int)blockIdx.y / args.slices;
    const int plane = lp & 1, l = lp >> 1;
    const uint16_t* reuse = args.reuse[plane];
    if (reuse == nullptr) return;
    const CUtensorMap* map = &maps.reuse[plane];
    uint16_t* out = args.out[plane];
    const Plane& rp = args.rp;
    const Plane& op = args.op;
    const int R = rp.chunks, n = rp.tokens, L = rp.layers;
    const int r = blockIdx.z % R, a0 = (blockIdx.z / R) * kAgentGroup;
    const int ag = min(kAgentGroup, args.agents - a0);
    const int D = rp.dim, half = D / 2, v8 = D / 8;
    const int HD = rp.heads * D, CW = kCW ? kCW : args.cw, c0 = slice * CW, P = CW / 8;
    const int b = args.b;
    const bool keys = plane == 0;
    const int tid = threadIdx.x, lane = tid & 31;
    const int rows = args.rows_per_cta;
    const int t_lo = blockIdx.x * rows, t_hi = min(n, t_lo + rows);
    const int TR = args.tile_rows;
    const MsLayout lay = ms_layout(CW, half, min(args.agents, kAgentGroup), rows, TR);
    uint16_t* ring = reinterpret_cast<uint16_t*>(smem + lay.ring);  // [stages][TR][CW]
    float* mu_s = reinterpret_cast<float*>(smem + lay.mu);
    float2* cs = reinterpret_cast<float2*>(smem + lay.cs);
    uint32_t* member = reinterpret_cast<uint32_t*>(smem + lay.member);
    float* wts = reinterpret_cast<float*>(smem + lay.wts);
    const unsigned tile_bytes = (unsigned)TR * CW * 2u;  // a box is always copied whole
    const int tiles = (t_hi - t_lo + TR - 1) / TR;
    int issued = 0;  // thread 0 only
    auto issue = [&](int k) {
        const int slot = k % kMsStages;
        mbar_arrive_expect_tx(&full[slot], tile_bytes);
        tma_load_4d(ring + (size_t)slot * TR * CW, map, c0, t_lo + k * TR, l, r, &full[slot]);
    };
    if (smem_u32(ring) & 127u) {  // never expected: report it instead of copying
        if (tid == 0) atomicOr(&g_status_repair, FLAG_INTERNAL);
        return;
    }
    if (tid == 0) {
        prefetch_tensormap(map);
        for (int q = 0; q < kMsStages; ++q) {
            mbar_init(&full[q], 1);
            mbar_init(&empty[q], kMsWarps);
        }
        fence_mbar_init();
        abort_flag = 0;
        // reused rows depend on no kernel of the chain: the first tiles go out at once
        for (; issued < min(kMsStages, tiles); ++issued) issue(issued);
    }
    for (int i = tid; i < ag * half; i += kMsThreads) {
        const int a = i / half, e = i % half;
        float c = 1.f, s = 0.f;
        if (keys) rope_cos_sin(args.delta[(a0 + a) * R + r], args.th.theta[e], &c, &s);
        cs[a * half + e] = make_float2(c, s);
    }
    if (tid < ag) rot_on[tid] = keys && args.delta[(a0 + tid) * R + r] != 0;
    for (int i = tid; i < ag * lay.words; i += kMsThreads) member[i] = 0u;
    pdl_wait();  // means (and, before them, probe sets and weights)
    __syncthreads();
    for (int i = tid; i < ag * CW; i += kMsThreads) {
        const int a = i / CW, e = i % CW;
        const long long u = (long long)(a0 + a) * R + r;
        mu_s[i] = args.mu[plane][(u * L + l) * HD + c0 + e];
    }
    if (b > 0) {
        for (int i = tid; i < ag * b; i += kMsThreads) {
            const int a = i / b;
            const long long u = (long long)(a0 + a) * R + r;
            const int j = args.idx[plane][u * b + (i % b)];
            if (j >= t_lo && j < t_hi) atomicOr(&member[a * lay.words + ((j - t_lo) >> 5)], 1u << ((j - t_lo) & 31));
        }
        for (int i = tid; i < ag * (t_hi - t_lo); i += kMsThreads) {
            const int a = i / (t_hi - t_lo), t = i % (t_hi - t_lo);
            const long long u = (long long)(a0 + a) * R + r;
            wts[a * rows + t] = args.w[plane][u * n + t_lo + t];
        }
    }
    __syncthreads();
    const int rpp = kMsThreads / P;  // rows per pass (P = cw / 8 divides the block)
    const int pq = tid % P, row_off = tid / P;
    const int h = pq / v8, v = pq % v8;
    const int eo = h * D + 4 * v;  // within the slice
    const long long pass_st = (long long)rpp * op.st;
    McConst kc;
    int cached = -1;  // agent whose constants sit in kc
    for (int k = 0; k < tiles; ++k) {
        const int slot = k % kMsStages;
        const unsigned parity = (unsigned)(k / kMsStages) & 1u;
        if (!mbar_wait(&full[slot], parity)) {
            atomicOr(&g_status_repair, FLAG_TIMEOUT);
            abort_flag = 1;
        }
        if (abort_flag) break;
        const uint16_t* tb = ring + (size_t)slot * TR * CW + eo;
        const int t0 = t_lo + k * TR;
        const int tt = min(TR, t_hi - t0);
        for (int a = 0; a < ag; ++a) {
            const bool rot = rot_on[a];
            if (a != cached) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const float2 ca = cs[a * half + 4 * v + 2 * q], cb = cs[a * half + 4 * v + 2 * q + 1];
                    kc.c2[q] = make_float2(ca.x, cb.x);
                    kc.s2[q] = make_float2(ca.y, cb.y);
                    kc.ns2[q] = make_float2(-ca.y, -cb.y);
                    const float* mm = mu_s + a * CW + eo + 2 * q;
                    kc.m0[q] = make_float2(mm[0], mm[1]);
                    kc.m1[q] = make_float2(mm[half], mm[half + 1]);
                }
                cached = a;
            }
            const long long u = (long long)(a0 + a) * R + r;
            const float* wb = wts + a * rows - t_lo;
            const uint32_t* mem = member + a * lay.words;
            uint16_t* o = out + op.row((int)u, l, t0 + row_off) + c0 + eo;
            if (kCW != 0 && kMsTileBytes / (2 * kCW) <= 64) {
                // TR <= 64 and tiles start at multiples of TR: the tile's probe bits are one
                // 64-bit window, and the row loop unrolls over the passes
                constexpr int kPasses = kCW ? (kMsTileBytes / (2 * kCW)) / (kMsThreads / (kCW / 8)) : 1;
                const int tl0 = t0 - t_lo;
                uint64_t pbits = 0;
                if (b > 0) {
                    const int w0 = tl0 >> 5, sh = tl0 & 31;
                    const uint64_t lo = mem[w0];
                    const uint64_t hi = (w0 + 1 < lay.words) ? mem[w0 + 1] : 0u;
                    const uint64_t x2 = (sh && w0 + 2 < lay.words) ? mem[w0 + 2] : 0u;
                    pbits = ((lo | (hi << 32)) >> sh) | (sh ? (x2 << (64 - sh)) : 0u);
                }
#pragma unroll
                for (int ps = 0; ps < kPasses; ++ps) {
                    const int row = row_off + ps * (kMsThreads / (kCW / 8));
                    if (row < tt && !((pbits >> row) & 1u))
                        correct_quad_pair(tb + row * kCW, o, half, rot, b > 0, b > 0 ? wb[t0 + row] : 0.f, kc);
                    o += pass_st;
                }
            } else {
                for (int row = row_off; row < tt; row += rpp, o += pass_st) {
                    const int tl = t0 + row - t_lo;
                    if (b > 0 && ((mem[tl >> 5] >> (tl & 31)) & 1u)) continue;  // probe row: written already
                    correct_quad_pair(tb + row * CW, o, half, rot, b > 0, b > 0 ? wb[t0 + row] : 0.f, kc);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (tid == 0 && issued < tiles && !abort_flag) {
            // the stage is free once every warp released it; then refill it
            if (!mbar_wait(&empty[slot], parity)) {
                atomicOr(&g_status_repair, FLAG_TIMEOUT);
                abort_flag = 1;
            } else {
                issue(issued);
                ++issued;
            }
        }
    }
    __syncthreads();
    if (abort_flag && tid == 0)  // a wait ran out: copies still in flight are waited for (bounded)
        for (int k = max(0, issued - kMsStages); k < issued; ++k)
            mbar_wait(&full[k % kMsStages], (unsigned)(k / kMsStages) & 1u);
}
// =====================================================================================
// Rounds of several agents: the same two steps with a fan-out stream.
//   round_mean_kernel: one CTA per (unit, layer, plane) computes that unit's probe mean
//     into the mean output, all units at once.  Warp g takes slots 4g..4g+3 and folds
//     them into the group sum Q_g; the CTA adds Q_0..Q_7 in order -- the arithmetic of
//     the one-agent probe-mean kernel, element for element.  Fresh probe rows are copied
//     to the output.
//   round_stream_kernel: one CTA per (row block, layer, plane, reused chunk, agent group)
//     reads each reused row once, through a 3-stage ring of bulk-copied 32 KB tiles with
//     full/empty mbarriers, and writes the corrected row of every agent of the group.  A
//     thread is one (agent, quad pair): its rotation and mean stay in registers for the
//     whole row block.
// =====================================================================================
constexpr int kRmThreads = 256;
constexpr int kRsThreads = 1024;
constexpr int kRsRows = 128;  // rows per CTA of the stream kernel
constexpr int kRsStages = 3;  // tiles of reused rows in flight per CTA
constexpr int kRsTileBytes = 32768;  // a stage: 16 rows of an 8 x 128 row

__global__ void __launch_bounds__(kRmThreads, 4) round_mean_kernel(McArgs args) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float ct[kMaxHeadDim / 2], st[kMaxHeadDim / 2];
    const int u = blockIdx.x, plane = blockIdx.y & 1, l = blockIdx.y >> 1;
    const uint16_t* reuse = args.reuse[plane];
    if (reuse == nullptr) return;
    const uint16_t* fresh = args.fresh[plane];
    uint16_t* out = args.out[plane];
    const Plane& rp = args.rp;
    const Plane& fp = args.fp;
    const Plane& op = args.op;
    const int R = rp.chunks, r = u % R, n = rp.tokens, L = rp.layers;
    const int D = rp.dim, half = D / 2, v8 = D / 8;
    const int HD = rp.heads * D, P = rp.heads * v8;
    const int b = args.b;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float* Qs = reinterpret_cast<float*>(smem);  // [8 groups][HD]
    const int dlt = args.delta[u];
    const bool rot = plane == 0 && dlt != 0;
    if (rot)  // independent of the selection: before the wait
        for (int e = tid; e < half; e += kRmThreads) rope_cos_sin(dlt, args.th.theta[e], &ct[e], &st[e]);
    pdl_wait();  // probe sets of the selection kernel
    // The stream kernel is released only at the end (its large CTAs would otherwise sit
    // waiting on SMs this kernel's later CTAs need).
    float* mu_g = args.mu[plane] + ((long long)u * L + l) * HD;
    if (b == 0) {
        for (int e = tid; e < HD; e += kRmThreads) mu_g[e] = 0.f;
        return;
    }
    __syncthreads();
    const int32_t* S = args.idx[plane] + (long long)u * b;
    const int grp = warp;  // warp g folds slots 4g..4g+3
    for (int pq = lane; pq < P; pq += 32) {
        const int h = pq / v8, v = pq % v8;
        const long long eo = (long long)h * D + 4 * v;
        float q0[4], q1[4];
#pragma unroll
        for (int j4 = 0; j4 < kSlotsPerGroup; ++j4) {
            const int s = grp * kSlotsPerGroup + j4;
            float fs0[4], fs1[4], xs0[4], xs1[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) fs0[k] = fs1[k] = xs0[k] = xs1[k] = 0.f;
            // two probe rows of the slot in flight at a time, summed in list order
            for (int i = s; i < b; i += 64) {
                const int j0 = __ldg(S + i), j1 = i + 32 < b ? __ldg(S + i + 32) : -2;
                uint2 xv[2][2], fv[2][2];
                bool ok[2];
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const int j = w ? j1 : j0;
                    ok[w] = j >= 0 && j < n;
                    if (!ok[w] && j != -2) atomicOr(&g_status_repair, FLAG_BOUNDS);
                    if (ok[w]) {
                        const long long ro = rp.row(r, l, j) + eo;
                        const long long fo = fp.row(u, l, j) + eo;
                        xv[w][0] = __ldg(reinterpret_cast<const uint2*>(reuse + ro));
                        xv[w][1] = __ldg(reinterpret_cast<const uint2*>(reuse + ro + half));
                        fv[w][0] = __ldcs(reinterpret_cast<const uint2*>(fresh + fo));
                        fv[w][1] = __ldcs(reinterpret_cast<const uint2*>(fresh + fo + half));
                    }
                }
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    if (!ok[w]) continue;
                    const long long oo = op.row(u, l, w ? j1 : j0) + eo;
                    __stcs(reinterpret_cast<uint2*>(out + oo), fv[w][0]);
                    __stcs(reinterpret_cast<uint2*>(out + oo + half), fv[w][1]);
                    add4(xv[w][0], xs0);
                    add4(xv[w][1], xs1);
                    add4(fv[w][0], fs0);
                    add4(fv[w][1], fs1);
                }
            }
            if (rot) {
                float c[4], sn[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    c[k] = ct[4 * v + k];
                    sn[k] = st[4 * v + k];
                }
                rotate4(xs0, xs1, c, sn);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float p0 = fs0[k] - xs0[k], p1 = fs1[k] - xs1[k];
                q0[k] = j4 == 0 ? p0 : q0[k] + p0;
                q1[k] = j4 == 0 ? p1 : q1[k] + p1;
            }
        }
        float* Q = Qs + grp * HD + h * D + 4 * v;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            Q[k] = q0[k];
            Q[half + k] = q1[k];
        }
    }
    __syncthreads();
    for (int e = tid; e < HD; e += kRmThreads) {
        float sum = 0.f;
#pragma unroll
        for (int g = 0; g < kGroups; ++g) sum += Qs[g * HD + e];
        mu_g[e] = sum / (float)b;
    }
    pdl_trigger();
}

__global__ void __launch_bounds__(kRsThreads) round_stream_kernel(McArgs args, int tile_rows) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kRsStages], empty[kRsStages];
    __shared__ int abort_flag;
    const int plane = blockIdx.y & 1, l = blockIdx.y >> 1;
    const uint16_t* reuse = args.reuse[plane];
    if (reuse == nullptr) return;
    uint16_t* out = args.out[plane];
    const Plane& rp = args.rp;
    const Plane& op = args.op;
    const int R = rp.chunks, n = rp.tokens, L = rp.layers;
    const int r = blockIdx.z % R, a0 = (blockIdx.z / R) * kAgentGroup;
    const int ag = min(kAgentGroup, args.agents - a0);
    const int D = rp.dim, half = D / 2, v8 = D / 8;
    const int HD = rp.heads * D, P = rp.heads * v8;
    const int b = args.b;
    const int tid = threadIdx.x, lane = tid & 31;
    const int t_lo = blockIdx.x * kRsRows, t_hi = min(n, t_lo + kRsRows);
    const int words = kRsRows / 32;
    const int TR = tile_rows;
    uint16_t* ring = reinterpret_cast<uint16_t*>(smem);                         // [kRsStages][TR][HD]
    float* cs = reinterpret_cast<float*>(ring + (size_t)kRsStages * TR * HD);   // [ag][half] cos, [ag][half] sin
    uint32_t* member = reinterpret_cast<uint32_t*>(cs + 2 * kAgentGroup * half);  // [ag][words]
    float* wts = reinterpret_cast<float*>(member + kAgentGroup * words);        // [ag][kRsRows]
    const bool keys = plane == 0;
    const int tiles = (t_hi - t_lo + TR - 1) / TR;
    const bool rows_contig = rp.st == HD;
    const unsigned row_bytes = (unsigned)HD * 2u;
    int issued = 0;  // thread 0 only
    // thread 0: bulk copies of tile k's reused rows into its stage, counted in bytes
    auto issue = [&](int k) {
        const int slot = k % kRsStages;
        const int t0 = t_lo + k * TR, tt = min(TR, t_hi - t0);
        uint16_t* dst = ring + (size_t)slot * TR * HD;
        mbar_arrive_expect_tx(&full[slot], row_bytes * tt);
        if (rows_contig) {
            bulk_g2s(dst, reuse + rp.row(r, l, t0), row_bytes * tt, &full[slot]);
        } else {
            for (int q = 0; q < tt; ++q) bulk_g2s(dst + q * HD, reuse + rp.row(r, l, t0 + q), row_bytes, &full[slot]);
        }
    };
    if (tid == 0) {
        for (int q = 0; q < kRsStages; ++q) {
            mbar_init(&full[q], 1);
            mbar_init(&empty[q], kRsThreads / 32);
        }
        fence_mbar_init();
        abort_flag = 0;
        // reused rows depend on no kernel of the chain: the first tiles go out at once
        for (; issued < min(kRsStages, tiles); ++issued) issue(issued);
    }
    for (int i = tid; i < ag * half; i += kRsThreads) {
        const int a = i / half, e = i % half;
        const int dlt = args.delta[(a0 + a) * R + r];
        float c = 1.f, s = 0.f;
        if (keys && dlt != 0) rope_cos_sin(dlt, args.th.theta[e], &c, &s);
        cs[a * half + e] = c;
        cs[(kAgentGroup + a) * half + e] = s;
    }
    for (int i = tid; i < ag * words; i += kRsThreads) member[i] = 0u;
    __syncthreads();
    // Probe sets and weights come from the selection, which completed before the mean
    // kernel (this kernel's predecessor) passed its own wait: they are read before this
    // kernel's wait, through L2.
    if (b > 0) {
        for (int i = tid; i < ag * b; i += kRsThreads) {
            const int a = i / b;
            const int j = __ldcg(args.idx[plane] + (long long)((a0 + a) * R + r) * b + i % b);
            if (j >= t_lo && j < t_hi) atomicOr(&member[a * words + ((j - t_lo) >> 5)], 1u << ((j - t_lo) & 31));
        }
        for (int i = tid; i < ag * (t_hi - t_lo); i += kRsThreads) {
            const int a = i / (t_hi - t_lo), t = i % (t_hi - t_lo);
            wts[a * kRsRows + t] = __ldcg(args.w[plane] + (long long)((a0 + a) * R + r) * n + t_lo + t);
        }
    }
    pdl_wait();  // the means
    __syncthreads();
    const int per_row = ag * P, rpp = kRsThreads / per_row;
    const bool active = tid < rpp * per_row;
    const int a = (tid % per_row) / P, pq = tid % P, row_off = tid / per_row;
    const int u = (a0 + a) * R + r;
    const int h = pq / v8, v = pq % v8;
    const int eo = h * D + 4 * v;
    const bool rot = keys && args.delta[min(u, args.agents * R - 1)] != 0;
    // the same float-pair constants and arithmetic as the one-agent stream kernel
    McConst kc;
    if (active) {
        const float* mu_g = args.mu[plane] + ((long long)u * L + l) * HD + eo;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float* ct = cs + a * half + 4 * v + 2 * q;
            const float* st = cs + (kAgentGroup + a) * half + 4 * v + 2 * q;
            kc.c2[q] = make_float2(ct[0], ct[1]);
            kc.s2[q] = make_float2(st[0], st[1]);
            kc.ns2[q] = make_float2(-st[0], -st[1]);
            kc.m0[q] = make_float2(mu_g[2 * q], mu_g[2 * q + 1]);
            kc.m1[q] = make_float2(mu_g[half + 2 * q], mu_g[half + 2 * q + 1]);
        }
    }
    const uint32_t* mem = member + a * words;
    const float* wb = wts + a * kRsRows;
    uint16_t* ob = out + op.row(u, l, 0) + eo;
    for (int k = 0; k < tiles; ++k) {
        const int slot = k % kRsStages;
        const unsigned parity = (unsigned)(k / kRsStages) & 1u;
        if (!mbar_wait(&full[slot], parity)) {
            atomicOr(&g_status_repair, FLAG_TIMEOUT);
            abort_flag = 1;
        }
        if (abort_flag) break;
        const uint16_t* tb = ring + (size_t)slot * TR * HD + eo;
        const int t0 = t_lo + k * TR, tt = min(TR, t_hi - t0);
        if (active) {
            // probe bits of the tile's rows (TR <= 32: at most two bitmap words)
            const int tl0 = t0 - t_lo;
            uint64_t pbits = 0;
            if (b > 0) {
                pbits = mem[tl0 >> 5];
                if ((tl0 & 31) + TR > 32) pbits |= (uint64_t)mem[(tl0 >> 5) + 1] << 32;
                pbits >>= (tl0 & 31);
            }
            uint16_t* o = ob + (long long)(t0 + row_off) * op.st;
            const long long ostep = (long long)rpp * op.st;
            for (int row = row_off; row < tt; row += rpp, o += ostep) {
                if ((pbits >> row) & 1u) continue;  // probe row: written already
                correct_quad_pair(tb + row * HD, o, half, rot, b > 0, b > 0 ? wb[tl0 + row] : 0.f, kc);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (tid == 0 && issued < tiles && !abort_flag) {
            // the stage is free once every warp released it; then refill it
            if (!mbar_wait(&empty[slot], parity)) {
                atomicOr(&g_status_repair, FLAG_TIMEOUT);
                abort_flag = 1;
            } else {
                issue(issued);
                ++issued;
            }
        }
    }
    __syncthreads();
    if (abort_flag && tid == 0)  // a wait ran out: copies still in flight are waited for (bounded)
        for (int k = max(0, issued - kRsStages); k < issued; ++k)
            mbar_wait(&full[k % kRsStages], (unsigned)(k / kRsStages) & 1u);
}

cudaError_t launch_mean_correct(const McPlanes& pl, const kvfix_kv_desc& rd, const kvfix_kv_desc& fd,
                                const kvfix_kv_desc& od, int agents, const int32_t* delta,
                                const RopeTheta& th, int b, cudaStream_t s) {
    McArgs a;
    for (int q = 0; q < 2; ++q) {
        a.reuse[q] = pl.reuse[q];
        a.fresh[q] = pl.fresh[q];
        a.out[q] = pl.out[q];
        a.idx[q] = pl.idx[q];
        a.w[q] = pl.w[q];
        a.mu[q] = pl.mu[q];
    }
    a.rp = plane_of(rd);
    a.fp = plane_of(fd);
    a.op = plane_of(od);
    a.agents = agents;
    a.b = b;
    a.delta = delta;
    a.th = th;
    const int n = a.rp.tokens;
    if (agents == 0 || a.rp.chunks == 0 || a.rp.layers == 0 || n == 0) return cudaSuccess;
    const int HD = a.rp.heads * a.rp.dim;
    if (agents > 1 && kAgentGroup * (HD / 8) <= kRsThreads) {
        // a round of several agents: all probe means at once, then one fan-out stream
        const size_t mean_smem = (size_t)kGroups * HD * sizeof(float);
        cudaError_t e = cudaFuncSetAttribute(round_mean_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)mean_smem);
        if (e != cudaSuccess) return e;
        e = launch_chained(round_mean_kernel, dim3(agents * a.rp.chunks, 2 * a.rp.layers), dim3(kRmThreads),
                           mean_smem, s, a);
        if (e != cudaSuccess) return e;
        const int half = a.rp.dim / 2;
        const int tile_rows = max(1, min(32, kRsTileBytes / (2 * HD)));
        const size_t stream_smem = (size_t)kRsStages * tile_rows * HD * 2 +
                                   sizeof(float) * (2 * kAgentGroup * half + kAgentGroup * kRsRows) +
                                   sizeof(uint32_t) * kAgentGroup * (kRsRows / 32);
        e = cudaFuncSetAttribute(round_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)stream_smem);
        if (e != cudaSuccess) return e;
        const int groups = (agents + kAgentGroup - 1) / kAgentGroup;
        return launch_chained(round_stream_kernel, dim3((n + kRsRows - 1) / kRsRows, 2 * a.rp.layers,
                                                        a.rp.chunks * groups),
                              dim3(kRsThreads), stream_smem, s, a, tile_rows);
    }
    // column slices of whole heads, kMcSliceCols elements wide unless one head is wider
    int hs = 1;
    for (int d = a.rp.heads; d >= 1; --d)
        if (a.rp.heads % d == 0 && d * a.rp.dim <= kMcSliceCols) {
            hs = d;
            break;
        }
    a.cw = hs * a.rp.dim;
    a.slices = a.rp.heads / hs;
    const int groups = (agents + kAgentGroup - 1) / kAgentGroup;
    const long long units = (long long)agents * a.rp.chunks;
    if (2ll * a.rp.layers * a.slices > 65535 || (long long)a.rp.chunks * groups > 65535 || units > 65535)
        return cudaErrorInvalidConfiguration;
    // the means: one CTA per (unit, layer, plane, slice), a thread per (slot, quad pair)
    const int pm_threads = kSlots * (a.cw / 8);
    const size_t pm_smem = (size_t)kSlots * a.cw * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(probe_mean_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pm_smem);
    if (e != cudaSuccess) return e;
    e = launch_chained(probe_mean_kernel, dim3(a.slices, 2 * a.rp.layers, (unsigned)units), dim3(pm_threads), pm_smem,
                       s, a);
    if (e != cudaSuccess) return e;
    // the stream: tiles of (cw x tile_rows) elements, 16 KB or the block's rows
    a.rows_per_cta = min(kMsRows, n);
    a.tile_rows = min(kMsTileBytes / (2 * a.cw), (a.rows_per_cta + 7) / 8 * 8);
    const int ag = agents < kAgentGroup ? agents : kAgentGroup;
    const MsLayout lay = ms_layout(a.cw, a.rp.dim / 2, ag, a.rows_per_cta, a.tile_rows);
    const size_t smem = (size_t)lay.total;
    if (smem > 220 * 1024) return cudaErrorInvalidValue;  // shape beyond the kernel's shared memory
    McMaps maps;
    memset(&maps, 0, sizeof maps);
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    for (int q = 0; q < 2; ++q) {
        if (!a.reuse[q]) continue;
        cuuint64_t dims[4], strides[3];
        plane_map_strides(a.rp, dims, strides);
        cuuint32_t box[4] = {(cuuint32_t)a.cw, (cuuint32_t)a.tile_rows, 1, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        if (enc(&maps.reuse[q], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(a.reuse[q]), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    auto kernel = a.cw == 128 ? mean_stream_kernel<128> : mean_stream_kernel<0>;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((n + a.rows_per_cta - 1) / a.rows_per_cta, 2 * a.rp.layers * a.slices, a.rp.chunks * groups);
    return launch_chained(kernel, grid, dim3(kMsThreads), smem, s, maps, a);
}

}  // namespace kvfix
